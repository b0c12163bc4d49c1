"""Planted mistakes in the oracle must fail its pins (CPU only).

Each case rewrites one line of an oracle function (a plausible slip: a flipped mask, a dropped term,
a wrong index or sign), installs the mutant in the oracle module for the duration of the case, and
runs the pins that concern that function: at least one of them must fail. This shows the pins in
tests/test_oracle.py are tied to the arithmetic, not to whatever the oracle happens to compute. The
comparison with torch's float64 attention (tests/test_oracle_vs_library.py) must catch every mutation of
a function it covers as well.
"""
import inspect
import textwrap

import pytest

import oracle
import test_oracle as pins
import test_oracle_vs_library as lib

# (name, oracle function, original text, mutated text, pins that must catch it)
MUTATIONS = [
    ("flipped causal mask", "head_scores", "s = np.where(cols > rows, -np.inf, s)",
     "s = np.where(cols < rows, -np.inf, s)",
     [(pins.test_causal_row_zero_sees_key_zero, {}), (pins.test_golden_two_key_example, {"causal": True})]),
    ("dropped D in dS", "attention_bwd", "ds = p * (dp - D)", "ds = p * dp",
     [(pins.test_backward_matches_central_differences, {"causal": False, "N": 9, "d": 8}),
      (pins.test_gradient_sums, {"causal": False})]),
    ("missing scale in dQ", "attention_bwd", "dq[b, h] = scale * (ds @ k[b, hk])", "dq[b, h] = ds @ k[b, hk]",
     [(pins.test_backward_matches_central_differences, {"causal": True, "N": 9, "d": 8})]),
    ("untransposed P in dV", "attention_bwd", "dv[b, hk] += p.T @ do[b, h]", "dv[b, hk] += p @ do[b, h]",
     [(pins.test_backward_matches_central_differences, {"causal": True, "N": 9, "d": 8}),
      (pins.test_gradient_sums, {"causal": True})]),
    ("dK sign", "attention_bwd", "dk[b, hk] += scale * (ds.T @ q[b, h])", "dk[b, hk] -= scale * (ds.T @ q[b, h])",
     [(pins.test_golden_two_key_example, {"causal": False})]),
    ("LSE in base 2", "_softmax_rows", "lse = m + np.log(l)", "lse = m + np.log2(l)",
     [(pins.test_q_zero_is_uniform_attention, {"causal": False}), (pins.test_single_key, {})]),
    ("grouped heads read the wrong K/V head", "_kv_head", "return h // (H // Hkv)", "return h % Hkv",
     [(pins.test_grouped_heads_equal_repeated_heads, {"causal": False, "Hkv": 2}),
      (pins.test_paged_decode_grouped_heads_equal_repeated_heads, {})]),
    ("key padding off by one", "head_scores", "s = np.where(cols >= kv_len, -np.inf, s)",
     "s = np.where(cols > kv_len, -np.inf, s)",
     [(pins.test_key_padding_equals_truncated_keys, {"causal": False}),
      (pins.test_no_visible_key_gives_zero_output, {"causal": False})]),
    ("page row index", "paged_attention_fwd", "rows = keys % ps", "rows = (keys + 1) % ps",
     [(pins.test_paged_decode_with_all_queries_is_causal_attention, {"Hkv": 1})]),
    ("decode causal alignment", "paged_attention_fwd", "pos = (L - Mq + np.arange(Mq))[:, None]",
     "pos = (L - Mq - 1 + np.arange(Mq))[:, None]",
     [(pins.test_paged_decode_with_all_queries_is_causal_attention, {"Hkv": 2})]),
    ("merge weight sign", "split_merge", "w = np.exp(lse_parts - m0[None])", "w = np.exp(m0[None] - lse_parts)",
     [(pins.test_split_merge_recovers_full_attention, {"causal": False})]),
]


def _mutant(name, original, mutated):
    src = textwrap.dedent(inspect.getsource(getattr(oracle, name)))
    assert src.count(original) == 1, f"{name}: the line to mutate is not in the oracle"
    ns = {}
    exec(compile(src.replace(original, mutated), f"<mutant of oracle.{name}>", "exec"), oracle.__dict__, ns)
    return ns[name]


@pytest.mark.parametrize("what,fn,original,mutated,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(monkeypatch, what, fn, original, mutated, catchers):
    for pin, kwargs in catchers:  # every catcher passes on the real oracle
        pin(**kwargs)
    monkeypatch.setattr(oracle, fn, _mutant(fn, original, mutated))
    caught = 0
    for pin, kwargs in catchers:
        try:
            pin(**kwargs)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught += 1
    assert caught >= 1, f"no pin catches: {what}"


# The same planted mistakes against the library comparison alone (tests/test_oracle_vs_library.py): every
# mutation of a function that comparison covers must fail it too. The LSE base and the split merge are
# outside it (the library returns neither), so they are left to the pins above.
LIBRARY_CATCHERS = {
    "flipped causal mask": (lib.test_matches_library_attention, {"causal": True, "N": 77, "d": 32}),
    "dropped D in dS": (lib.test_matches_library_attention, {"causal": False, "N": 77, "d": 32}),
    "missing scale in dQ": (lib.test_matches_library_attention, {"causal": True, "N": 77, "d": 32}),
    "untransposed P in dV": (lib.test_matches_library_attention, {"causal": False, "N": 77, "d": 32}),
    "dK sign": (lib.test_matches_library_attention, {"causal": True, "N": 77, "d": 32}),
    "grouped heads read the wrong K/V head": (lib.test_grouped_heads_match_library, {"Hkv": 2, "causal": False}),
    "key padding off by one": (lib.test_key_padding_matches_library, {"causal": False}),
    "page row index": (lib.test_paged_decode_matches_library, {"causal": False}),
    "decode causal alignment": (lib.test_paged_decode_matches_library, {"causal": True}),
}


@pytest.mark.parametrize("what,fn,original,mutated", [m[:4] for m in MUTATIONS if m[0] in LIBRARY_CATCHERS],
                         ids=[m[0] for m in MUTATIONS if m[0] in LIBRARY_CATCHERS])
def test_planted_mistake_fails_the_library_comparison(monkeypatch, what, fn, original, mutated):
    pin, kwargs = LIBRARY_CATCHERS[what]
    pin(**kwargs)  # passes on the real oracle
    monkeypatch.setattr(oracle, fn, _mutant(fn, original, mutated))
    with pytest.raises((AssertionError, ValueError, IndexError, FloatingPointError)):
        pin(**kwargs)
