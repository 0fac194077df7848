"""Target / draft logits and drafted tokens for the speculative sampler.

Recipe: p_logits ~ N(0, p_sigma^2) fp32 for k+1
positions, q_logits = p_logits[:k] + N(0, q_sigma^2), drafted tokens
x_i ~ softmax(q_logits[i]) drawn by the Gumbel-max trick (argmax of logits
plus Gumbel noise), so no normalisation happens here.
"""

from dataclasses import dataclass

import torch


@dataclass
class SpecInputs:
    p_logits: torch.Tensor      # [N][k+1][V] float32
    q_logits: torch.Tensor      # [N][k][V] float32
    draft_tokens: torch.Tensor  # [N][k] int32


def make_spec_inputs(num_seqs, k, vocab, p_sigma, q_sigma, seed, device="cpu", chunk=64):
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    N, k, V = int(num_seqs), int(k), int(vocab)
    p = torch.empty((N, k + 1, V), dtype=torch.float32, device=device)
    q = torch.empty((N, k, V), dtype=torch.float32, device=device)
    x = torch.empty((N, k), dtype=torch.int32, device=device)
    for n0 in range(0, N, chunk):
        n1 = min(N, n0 + chunk)
        pc = torch.randn((n1 - n0, k + 1, V), generator=gen, device=device) * float(p_sigma)
        qc = pc[:, :k] + torch.randn((n1 - n0, k, V), generator=gen, device=device) * float(q_sigma)
        u = torch.rand((n1 - n0, k, V), generator=gen, device=device)
        gumbel = -torch.log(-torch.log(u.clamp_min(1e-38)))
        x[n0:n1] = torch.argmax(qc + gumbel, dim=-1).to(torch.int32)
        p[n0:n1] = pc
        q[n0:n1] = qc
    return SpecInputs(p_logits=p, q_logits=q, draft_tokens=x)
