"""Planted mistakes in the oracle are caught by its pins.

Each case rewrites one line of an oracle function (a dropped term, a wrong
sign, a swapped operand or index, the gate applied in the wrong place, a chunk
reset counted from the wrong token), installs the mutant in place of the
function for the duration of the case, and runs the pins of
tests/test_oracle_pins.py (the token recurrences, decode) or
tests/test_state_pass_pins.py (the chunk state pass, forward and backward): at
least one of them must fail on an assertion.  All on the CPU; the oracle
itself is never edited.
"""
import inspect
import textwrap

import pytest

import test_oracle_pins as P
from oracle import recurrence as R

# every pin, with the arguments of each of its parametrisations
PINS = [
    (P.test_hand_worked_example, {}),
    (P.test_recurrence_matches_transition_product, {"per_channel": False}),
    (P.test_recurrence_matches_transition_product, {"per_channel": True}),
    (P.test_beta_zero_gate_zero_keeps_state, {"per_channel": False}),
    (P.test_beta_zero_gate_zero_keeps_state, {"per_channel": True}),
    (P.test_delta_rule_writes_value_exactly, {}),
    (P.test_gate_to_minus_infinity_resets_state, {}),
    (P.test_kda_with_channel_constant_gate_equals_gdn, {}),
    (P.test_grouped_heads_equal_repeated_heads, {}),
    (P.test_varlen_equals_separate_runs_and_cumsum_gate_input, {}),
    (P.test_prefix_then_resume_equals_full_run, {}),
    (P.test_softplus_against_log1p_and_threshold_edge, {}),
    (P.test_decode_gates_closed_form, {}),
    (P.test_decode_matches_prefill_recurrence_and_chains_over_calls, {}),
    (P.test_l2_normalize_eps_inside_root, {}),
    (P.test_kda_cumsum_gate_input_equals_raw_and_transition_product, {"chunk": 4}),
    (P.test_kda_cumsum_gate_reset_counts_chunks_from_each_sequence_start, {}),
    (P.test_decode_without_l2norm_matches_transition_product, {}),
    (P.test_chunked_equals_recurrent_for_every_chunk_length, {"per_channel": False}),
    (P.test_chunked_equals_recurrent_for_every_chunk_length, {"per_channel": True}),
]

# (function, line as written, planted replacement)
MUTATIONS = {
    "gdn: gate dropped": ("gdn_recurrent", "S = math.exp(gg[t]) * S", "S = S"),
    "gdn: gate after the update": (
        "gdn_recurrent",
        "S = math.exp(gg[t]) * S",
        "pass",
        "S = S + np.outer(delta, kt)",
        "S = math.exp(gg[t]) * (S + np.outer(delta, kt))"),
    "gdn: wrong sign of the prediction": (
        "gdn_recurrent", "(v[b, t, h] - pred)", "(v[b, t, h] + pred)"),
    "gdn: beta dropped": (
        "gdn_recurrent", "delta = beta[b, t, h] * (v[b, t, h] - pred)",
        "delta = (v[b, t, h] - pred)"),
    "gdn: scale dropped": (
        "gdn_recurrent", "o[b, t, h] = scale * (S @ q[b, t, hk])", "o[b, t, h] = S @ q[b, t, hk]"),
    "gdn: output from the state before the token": (
        "gdn_recurrent",
        "S = S + np.outer(delta, kt)\n                o[b, t, h] = scale * (S @ q[b, t, hk])",
        "o[b, t, h] = scale * (S @ q[b, t, hk])\n                S = S + np.outer(delta, kt)"),
    "gdn: key head of a value head": ("gdn_recurrent", "hk = h // (H // Hg)", "hk = h % Hg"),
    "gdn: query in place of the key": ("gdn_recurrent", "pred = S @ kt", "pred = S @ q[b, t, hk]"),
    "gdn: initial state not transposed": (
        "gdn_recurrent", "h0[n, h].T.copy()", "h0[n, h].reshape(S_shape := (v.shape[3], k.shape[3]))"),
    "kda: channel gates averaged": (
        "kda_recurrent", "S = S * np.exp(gg[t])[None, :]", "S = S * np.exp(np.mean(gg[t]))"),
    "kda: wrong sign of the prediction": (
        "kda_recurrent", "(v[b, t, hv] - pred)", "(v[b, t, hv] + pred)"),
    "kda: gate after the update": (
        "kda_recurrent",
        "S = S * np.exp(gg[t])[None, :]",
        "pass",
        "S = S + np.outer(delta, kt)",
        "S = (S + np.outer(delta, kt)) * np.exp(gg[t])[None, :]"),
    "cumsum gate: chunks counted from token 0": (
        "raw_gate_from_chunk_cumsum", "(t - bos) % chunk_size != 0", "t % chunk_size != 0"),
    "cumsum gate: no reset at chunk starts": (
        "raw_gate_from_chunk_cumsum", "(t - bos) % chunk_size != 0", "t != bos"),
    "decode: gate after the update": (
        "gdn_decode",
        "S = math.exp(g[bi, t, hv]) * S",
        "pass",
        "S = S + np.outer(delta, kn[bi, t, hk])",
        "S = math.exp(g[bi, t, hv]) * (S + np.outer(delta, kn[bi, t, hk]))"),
    "decode: query not scaled": ("gdn_decode", "qn = l2_normalize(q, eps) * scale", "qn = l2_normalize(q, eps)"),
    "decode gates: decay sign": (
        "decode_gates", "g = -np.exp(A_log)[None, None, :]", "g = np.exp(A_log)[None, None, :]"),
    "decode gates: beta not a sigmoid": (
        "decode_gates", "beta = 1.0 / (1.0 + np.exp(-b))", "beta = 1.0 / (1.0 + np.exp(b))"),
    "softplus: threshold test reversed": ("softplus", "bx <= threshold", "bx > threshold"),
    "l2 norm: eps outside the root": (
        "l2_normalize", "np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)",
        "(np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)"),
}


def _mutant(name, *edits):
    fn = getattr(R, name)
    src = textwrap.dedent(inspect.getsource(fn))
    for old, new in zip(edits[::2], edits[1::2]):
        assert src.count(old) == 1, f"{name}: {old!r} is not one line of the oracle"
        src = src.replace(old, new)
    ns = dict(vars(R))
    exec(compile(src, f"<mutant of {name}>", "exec"), ns)
    return ns[name]


@pytest.mark.parametrize("case", list(MUTATIONS))
def test_planted_mistake_fails_a_pin(case, monkeypatch):
    name, *edits = MUTATIONS[case]
    monkeypatch.setattr(R, name, _mutant(name, *edits))
    for pin, kwargs in PINS:
        try:
            pin(**kwargs)
        except AssertionError:  # a pin saw wrong values (a mutant that cannot run fails the case)
            return
    pytest.fail(f"no pin fails with the planted mistake: {case}")


# ---- the chunk state pass (forward and backward) and its pins ----------------

import test_state_pass_pins as SPP  # noqa: E402
from oracle import state_pass as SP  # noqa: E402

SP_PINS = (
    [(SPP.test_final_state_matches_closed_form, {"gate": g}) for g in SP.GATES]
    + [(SPP.test_gate_kinds_reduce_to_each_other, {}),
       (SPP.test_chunk_starts_resume_the_run_and_packed_sequences_are_separate_runs, {})]
    + [(SPP.test_state_gradient_is_the_adjoint_of_the_forward_pass, {"gate": g}) for g in SP.GATES]
    + [(SPP.test_state_gradient_grouped_query_heads_share_the_gate, {}),
       (SPP.test_split_size_keeps_every_split_chunk, {"split": 128}),
       (SPP.test_state_v_first_transposes_every_state, {})])

SP_MUTATIONS = {
    "state: per-key gate averaged over the keys": (
        "chunk_state_pass", "S = np.exp(raw[t, h])[:, None] * S", "S = np.exp(raw[t, h].mean()) * S"),
    "state: per-value gate averaged over the values": (
        "chunk_state_pass", "S = S * np.exp(raw[t, h])[None, :]", "S = S * np.exp(raw[t, h].mean())"),
    "state: per-head rate with the wrong sign": (
        "chunk_state_pass", "S = np.exp(gv_[h]) * S", "S = np.exp(-gv_[h]) * S"),
    "state: update subtracted": (
        "chunk_state_pass", "S = S + np.outer(k[b, t, h], v[b, t, h])",
        "S = S - np.outer(k[b, t, h], v[b, t, h])"),
    "state: scalar gate after the update": (
        "chunk_state_pass",
        "S = np.exp(raw[t, h]) * S", "pass",
        "S = S + np.outer(k[b, t, h], v[b, t, h])",
        "S = (np.exp(raw[t, h]) if gate == 'g' else 1.0) * (S + np.outer(k[b, t, h], v[b, t, h]))"),
    "state: chunk-start state one token late": (
        "chunk_state_pass", "if i % chunk_size == 0 and", "if i % chunk_size == 1 and"),
    "grad: scale dropped": (
        "chunk_state_grad", "G = G + scale * np.outer(q[b, t, hq], do[b, t, hq])",
        "G = G + np.outer(q[b, t, hq], do[b, t, hq])"),
    "grad: output term with the wrong sign": (
        "chunk_state_grad", "G = G + scale * np.outer(q[b, t, hq], do[b, t, hq])",
        "G = G - scale * np.outer(q[b, t, hq], do[b, t, hq])"),
    "grad: scalar gate before the output term": (
        "chunk_state_grad",
        "G = G + scale * np.outer(q[b, t, hq], do[b, t, hq])", "pass",
        "G = np.exp(raw[t, h]) * G",
        "G = np.exp(raw[t, h]) * G + scale * np.outer(q[b, t, hq], do[b, t, hq])"),
    "grad: wrong gate head of a query head": ("chunk_state_grad", "h = hq // group", "h = hq % H"),
    "grad: chunk gradient stored at the chunk's start": (
        "chunk_state_grad", "i % chunk_size == chunk_size - 1 or", "i % chunk_size == 0 or"),
}


def _sp_mutant(name, *edits):
    fn = getattr(SP, name)
    src = textwrap.dedent(inspect.getsource(fn))
    for old, new in zip(edits[::2], edits[1::2]):
        assert src.count(old) == 1, f"{name}: {old!r} is not one line of the oracle"
        src = src.replace(old, new)
    ns = dict(vars(SP))
    exec(compile(src, f"<mutant of {name}>", "exec"), ns)
    return ns[name]


@pytest.mark.parametrize("case", list(SP_MUTATIONS))
def test_planted_state_pass_mistake_fails_a_pin(case, monkeypatch):
    name, *edits = SP_MUTATIONS[case]
    monkeypatch.setattr(SP, name, _sp_mutant(name, *edits))
    for pin, kwargs in SP_PINS:
        try:
            pin(**kwargs)
        except AssertionError:
            return
    pytest.fail(f"no pin fails with the planted mistake: {case}")
