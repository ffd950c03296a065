"""Planted controls: copies of the oracle with one mistake each must fail the
pins. The pages' kernel contract plants four such controls (PR #1377 "LFM2:
shared-round decode", its kernel-contract commit): a pick that takes the
highest id on a tie, a row with a nonfinite logit left unflagged, and all
streams sharing stream 0's conv state or KV cache (for reads or writes); the
rest guard the readings the pins fix. The draft side's controls follow the
pages' drafter contract (PR #1391 "lfm2: draft with LiquidAI's DSpark
drafter", the commit adding controls for the Markov head, the draft ids and
the block attention): a NaN score left unflagged, all streams taking stream
0's previous token, a pick beyond the vocabulary kept as a token, a block row
that misses the last key.
The mistakes are planted in the oracle's source, on the CPU.
"""

import inspect
import types

import pytest

import oracle.draft as oracle_draft
import oracle.step as oracle_step
import oracle_pins as P
import oracle_pins_draft as PD


def mutant(*edits, module=oracle_step):
    src = inspect.getsource(module)
    src = src.replace("from .step import", "from oracle.step import")
    for old, new in edits:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


CONTROLS = {
    "tie_to_highest_id": (
        [("pick[r] = int(np.argmax(row))  # first occurrence of the maximum",
          "pick[r] = int(len(row) - 1 - np.argmax(row[::-1]))")],
        [P.pin_argmax_golden, P.pin_argmax_brute]),
    "nonfinite_not_flagged": (
        [("if not np.all(np.isfinite(row)):", "if False:")],
        [P.pin_argmax_golden]),
    "streams_read_first_conv_state": (
        [("short_conv_stream(bcx[off:off + rows], w, states[s], want_history)",
          "short_conv_stream(bcx[off:off + rows], w, states[0], want_history)")],
        [P.pin_segmented_equals_alone]),
    "streams_write_first_conv_state": (
        [("        new_states.append(st)\n", "        new_states[0:1] = [st]\n")],
        [P.pin_segmented_equals_alone]),
    "streams_read_first_kv_cache": (
        [("attention_stream(q[off:off + rows], Ks[s], Vs[s], keys, rows, full)",
          "attention_stream(q[off:off + rows], Ks[0], Vs[0], keys, rows, full)")],
        [P.pin_segmented_equals_alone]),
    "conv_taps_reversed": (
        [("conv = (wf[:, 0] * bf16_to_f64(seq[i])", "conv = (wf[:, 2] * bf16_to_f64(seq[i])"),
         ("+ wf[:, 2] * bf16_to_f64(seq[i + 2]))", "+ wf[:, 0] * bf16_to_f64(seq[i + 2]))")],
        [P.pin_conv_worked]),
    "gate_truncated": (
        [("return (upper + up.astype(np.uint64)).astype(np.uint16)", "return upper.astype(np.uint16)")],
        [P.pin_bf16_rounding_golden, P.pin_conv_worked, P.pin_bf16_rounding_matches_torch]),
    "conv_slices_swapped": (
        [("c = bf16_to_f64(bcx[i, h:2 * h])", "c = bf16_to_f64(bcx[i, 2 * h:3 * h])"),
         ("x = bf16_to_f64(bcx[i, 2 * h:3 * h])", "x = bf16_to_f64(bcx[i, h:2 * h])")],
        [P.pin_conv_worked, P.pin_conv_special_taps]),
    "score_not_scaled": (
        [("SCALE = 0.125 ", "SCALE = 1.0 ")],
        [P.pin_attn_two_keys_scale, P.pin_attn_brute]),
    "causal_off_by_one": (
        [("return keys - rows + i + 1", "return keys - rows + i + 2")],
        [P.pin_attn_one_key, P.pin_attn_causal_edge]),
    "gqa_mapping_wrong": (
        [("            g = h // GROUP\n", "            g = h % NKV\n")],
        [P.pin_attn_gqa]),
    "merge_sums_unrescaled_l": (
        [("L = (wgt * l).sum(axis=-1)", "L = l.sum(axis=-1)")],
        [P.pin_attn_split_merge]),
    "accept_compares_next_pick": (
        [("or flag[a] or int(pick[a]) != d:", "or flag[a] or int(pick[a + 1]) != d:")],
        [P.pin_accept_cases, P.pin_accept_recipe]),
    "rewind_one_row_early": (
        [("return np.stack([history[a + 1], history[a + 2]])", "return np.stack([history[a], history[a + 1]])")],
        [P.pin_rewind]),
    "block_row_missing_last_key": (
        [("    if full:\n        return keys\n", "    if full:\n        return keys - 1\n")],
        [P.pin_attn_full_q_zero, P.pin_attn_full_brute]),
    "block_rows_causal": (
        [("    if full:\n        return keys\n", "    if False:\n        return keys\n")],
        [P.pin_attn_full_q_zero, P.pin_attn_full_split_merge]),
}

DRAFT_CONTROLS = {
    "markov_nan_score_not_flagged": (
        [("    if not np.all(np.isfinite(score)):\n", "    if False:\n")],
        [PD.pin_markov_worked]),
    "markov_tie_to_highest_token": (
        [("int(np.argmax(score))", "int(len(score) - 1 - np.argmax(score[::-1]))")],
        [PD.pin_markov_worked]),
    "markov_chain_stuck_on_pending_token": (
        [("        prev = p\n", "")],
        [PD.pin_markov_worked, PD.pin_markov_permutation_chain]),
    "markov_dot_not_rounded": (
        [("dot16 = bf16_to_f64(f64_to_bf16_rne_any(dot))", "dot16 = dot")],
        [PD.pin_markov_worked, PD.pin_markov_brute]),
    "markov_w2_column_for_row": (
        [("dot = bf16_to_f64(W2) @ e", "dot = bf16_to_f64(W2).T[:, :len(e)] @ e if W2.shape[0] == W2.shape[1] else bf16_to_f64(W2) @ e")],
        [PD.pin_markov_permutation_chain]),
    "markov_streams_read_first_pending_token": (
        [("markov_chain(base[b:b + rows - 1], W1, W2, prev[s])", "markov_chain(base[b:b + rows - 1], W1, W2, prev[0])")],
        [PD.pin_markov_streams]),
    "rounding_through_binary32": (
        [("r = np.rint(v / quantum) * quantum", "r = np.rint(float(np.float32(v)) / quantum) * quantum")],
        [PD.pin_bf16_any_golden, PD.pin_bf16_any_brute]),
    "draft_ids_streams_read_first_pending_token": (
        [("p = int(prev[s])", "p = int(prev[0])")],
        [PD.pin_draft_ids_golden]),
    "draft_ids_pick_past_vocab_keeps_token": (
        [("bad = (draft_flag is not None and draft_flag[k]) or not (0 <= d < vocab)",
          "bad = draft_flag is not None and draft_flag[k]")],
        [PD.pin_draft_ids_golden]),
    "draft_ids_flagged_pick_copied": (
        [("bad = (draft_flag is not None and draft_flag[k]) or not (0 <= d < vocab)",
          "bad = not (0 <= d < vocab)")],
        [PD.pin_draft_ids_golden]),
}


@pytest.mark.parametrize("name", sorted(CONTROLS))
def test_planted_control_goes_red(name):
    edits, pins = CONTROLS[name]
    mod = mutant(*edits)
    for pin in pins:
        with pytest.raises(Exception):
            pin(mod)


@pytest.mark.parametrize("name", sorted(DRAFT_CONTROLS))
def test_planted_draft_control_goes_red(name):
    edits, pins = DRAFT_CONTROLS[name]
    mod = mutant(*edits, module=oracle_draft)
    for pin in pins:
        with pytest.raises(Exception):
            pin(mod)
