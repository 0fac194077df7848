"""Pin of the oracle's Philox4x32-10 against CUDA's curand implementation of
the same generator (Salmon et al., SC'11): raw 32-bit outputs must agree bit
for bit on random and edge-case counters and keys."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from probes import build_probes

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_oracle_philox_equals_curand_device_routine():
    lib = ctypes.CDLL(build_probes.build())
    rng = np.random.default_rng(2024)
    n = 1 << 16
    ctr = rng.integers(0, 1 << 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 1 << 32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    # edge cases: all-zero, all-ones, and the sampler's own counter layout
    ctr[0], key[0] = 0, 0
    ctr[1], key[1] = 0xFFFFFFFF, 0xFFFFFFFF
    ctr[2:10] = np.array([[s, p, st, 7] for s in (0, 2047) for p in (0, 8) for st in (0, 1)], dtype=np.uint32)
    key[2:10] = [0, 0]
    d_ctr = torch.from_numpy(ctr.view(np.int32)).to(DEV)
    d_key = torch.from_numpy(key.view(np.int32)).to(DEV)
    d_out = torch.empty((n, 4), dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.philox_probe_run(ctypes.c_void_p(d_ctr.data_ptr()), ctypes.c_void_p(d_key.data_ptr()),
                              ctypes.c_void_p(d_out.data_ptr()), ctypes.c_int(n), stream)
    assert rc == 0
    got = d_out.cpu().numpy().view(np.uint32)
    want = np.stack(oracle.philox4x32_10(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3], key[:, 0], key[:, 1]),
                    axis=1)
    assert np.array_equal(got, want)
