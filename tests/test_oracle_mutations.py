"""The oracle's pins are strong enough: a plausible mistake planted in the
oracle (a dropped term, a wrong sign, an off-by-one index, a swapped operand)
makes at least one pin fail.  Mutations are planted on the CPU only, by
rewriting one line of an oracle function's source and patching the result in
for the duration of a test."""

import inspect
import sys
import textwrap

import pytest

import oracle.attention as oatt
import oracle.draft_sample as odraft
import oracle.kv_cache as okv
import oracle.scheduler as osched
import oracle.philox as ophil
import oracle.selection as osel
import oracle as oracle_pkg
import oracle.spec_sample  # noqa: F401  (the package re-exports a function of the same name)
import test_oracle_attention as pins_att
import test_oracle_draft_sample as pins_draft
import test_oracle_kv_cache as pins_kv
import test_oracle_scheduler as pins_sched
import test_oracle_philox as pins_phil
import test_oracle_select as pins_sel
import test_oracle_spec_sample as pins_spec

ospec = sys.modules["oracle.spec_sample"]


def _mutant(module, func_name, old, new):
    """A copy of module.func_name with the source text `old` replaced by `new`."""
    src = textwrap.dedent(inspect.getsource(getattr(module, func_name)))
    assert src.count(old) == 1, f"mutation anchor not found once in {func_name}: {old!r}"
    ns = dict(module.__dict__)
    exec(compile(src.replace(old, new), f"<mutant of {func_name}>", "exec"), ns)
    return ns[func_name]


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


def test_dropped_softmax_scale_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "_attend", _mutant(oatt, "_attend", "sm_scale * (keys @ qvec)", "(keys @ qvec)"))
    _fails(pins_att.test_dense_matches_library_attention, 0.37)


def test_keys_used_as_values_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "_attend", _mutant(oatt, "_attend", "return w @ values, w", "return w @ keys, w"))
    _fails(pins_att.test_closed_forms)


def test_missing_max_subtraction_is_harmless_but_missing_normalisation_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "_attend", _mutant(oatt, "_attend", "w = e / e.sum()", "w = e"))
    _fails(pins_att.test_closed_forms)


def test_causal_off_by_one_in_verify_is_caught(monkeypatch):
    mutant = _mutant(oatt, "verify_attn", "visible = L + i + 1", "visible = L + i")
    monkeypatch.setattr(pins_att, "verify_attn", mutant)
    _fails(pins_att.test_verify_rows_equal_sequential_decodes)
    _fails(pins_att.test_verify_matches_library_causal_attention_and_mass)


def test_draft_tail_off_by_one_is_caught(monkeypatch):
    mutant = _mutant(oatt, "draft_visible_tokens", "L + int(draft_pos) + 1", "L + int(draft_pos)")
    monkeypatch.setattr(oatt, "draft_visible_tokens", mutant)
    _fails(pins_att.test_budget_one_sparse_equals_dense)


def test_wrong_gqa_group_mapping_is_caught(monkeypatch):
    mutant = _mutant(oatt, "dense_decode_attn", "qh = h * G + g", "qh = g * Hkv + h")
    monkeypatch.setattr(pins_att, "dense_decode_attn", mutant)
    _fails(pins_att.test_gqa_mapping_uses_contiguous_groups)


def test_page_mass_on_wrong_page_is_caught(monkeypatch):
    mutant = _mutant(oatt, "verify_attn", "tokens[:visible] // PAGE_SIZE", "(tokens[:visible] + 1) // PAGE_SIZE")
    monkeypatch.setattr(pins_att, "verify_attn", mutant)
    _fails(pins_att.test_verify_matches_library_causal_attention_and_mass)


def test_reversed_tie_break_in_selection_is_caught(monkeypatch):
    mutant = _mutant(osel, "select_draft_pages", "key=lambda pg: (-mass[s, h, pg], pg)",
                     "key=lambda pg: (-mass[s, h, pg], -pg)")
    monkeypatch.setattr(pins_sel, "select_draft_pages", mutant)
    _fails(pins_sel.test_matches_brute_force_with_ties, 0)


def test_budget_without_mandatory_floor_is_caught(monkeypatch):
    mutant = _mutant(osel, "selection_budget", "max(math.ceil(float(budget) * P - 1e-9), len(mandatory))",
                     "math.ceil(float(budget) * P - 1e-9)")
    monkeypatch.setattr(osel, "selection_budget", mutant)
    monkeypatch.setattr(pins_sel, "selection_budget", mutant, raising=False)
    _fails(pins_sel.test_budget_arithmetic)


def test_wrong_philox_multiplier_is_caught(monkeypatch):
    monkeypatch.setattr(ophil, "M0", 0xD2511F55)
    _fails(pins_phil.test_known_answer_vectors)


def test_missing_key_bump_in_philox_is_caught(monkeypatch):
    mutant = _mutant(ophil, "philox4x32_10", "k0 = (k0 + np.uint64(W0)) & np.uint64(MASK32)", "k0 = k0")
    monkeypatch.setattr(pins_phil, "philox4x32_10", mutant)
    _fails(pins_phil.test_known_answer_vectors)


def test_residual_with_wrong_sign_is_caught(monkeypatch):
    mutant = _mutant(ospec, "spec_sample", "r = np.maximum(p[pn[rej], i] - q[qn[rej], i], 0.0)",
                     "r = np.maximum(q[qn[rej], i] - p[pn[rej], i], 0.0)")
    monkeypatch.setattr(pins_spec, "spec_sample", mutant)
    _fails(pins_spec.test_output_distribution_equals_target)


def test_bonus_from_the_draft_row_is_caught(monkeypatch):
    mutant = _mutant(ospec, "spec_sample", "row[~rej] = p[pn[~rej], k]", "row[~rej] = q[qn[~rej], k - 1]")
    monkeypatch.setattr(pins_spec, "spec_sample", mutant)
    _fails(pins_spec.test_output_distribution_equals_target)


def test_draft_sampler_on_the_wrong_stream_is_caught(monkeypatch):
    mutant = _mutant(odraft, "sample_draft_tokens", "int(draft_pos), STREAM_DRAFT)", "int(draft_pos), 1)")
    monkeypatch.setattr(pins_draft, "sample_draft_tokens", mutant)
    _fails(pins_draft.test_uniform_logits_give_floor_u_times_v)


def test_append_into_the_next_slot_is_caught(monkeypatch):
    mutant = _mutant(okv, "kv_append", "k_out[page, :, pos % PAGE_SIZE, :] = k_rows[s, t]",
                     "k_out[page, :, (pos + 1) % PAGE_SIZE, :] = k_rows[s, t]")
    monkeypatch.setattr(pins_kv, "kv_append", mutant)
    _fails(pins_kv.test_append_reads_back_through_whole_page_rebuild)


def test_commit_without_the_pending_token_is_caught(monkeypatch):
    mutant = _mutant(okv, "commit_lengths", "np.asarray(n_accepted, dtype=np.int64) + 1",
                     "np.asarray(n_accepted, dtype=np.int64)")
    monkeypatch.setattr(pins_kv, "commit_lengths", mutant)
    _fails(pins_kv.test_commit_closed_form)


def test_aimd_blind_to_the_backlog_is_caught(monkeypatch):
    mutant = _mutant(osched, "simulate", 'if util > cfg["util_high"] or len(paused) > cfg["backlog_max"]:',
                     'if util > cfg["util_high"]:')
    monkeypatch.setattr(pins_sched, "simulate", mutant)
    _fails(pins_sched.test_multiplicative_cut_closed_form)


def test_new_requests_ahead_of_paused_ones_is_caught(monkeypatch):
    mutant = _mutant(osched, "simulate", "            if paused:\n", "            if paused and not waiting:\n")
    monkeypatch.setattr(pins_sched, "simulate", mutant)
    _fails(pins_sched.test_invariants_on_random_workloads, osched.POLICY_AIMD, 1)


def test_tie_judge_residual_with_wrong_sign_is_caught(monkeypatch):
    mutant = _mutant(ospec, "residual_row", "r = np.maximum(p - q, 0.0)", "r = np.maximum(q - p, 0.0)")
    monkeypatch.setattr(ospec, "residual_row", mutant)
    monkeypatch.setattr(oracle_pkg, "residual_row", mutant)
    _fails(pins_spec.test_residual_of_disjoint_supports_is_the_target)


def test_tie_judge_residual_without_fallback_is_caught(monkeypatch):
    mutant = _mutant(ospec, "residual_row", "        return p\n", "        return r\n")
    monkeypatch.setattr(ospec, "residual_row", mutant)
    monkeypatch.setattr(oracle_pkg, "residual_row", mutant)
    _fails(pins_spec.test_residual_of_equal_rows_falls_back_to_the_target)
