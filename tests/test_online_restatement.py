"""The tiled online-softmax algorithm (fp64 restatement) reaches the oracle's
three-step result, the split-KV combine does too, and the parity gate rejects
planted mistakes in the algorithm while admitting a 16-bit-rounded run of it."""
import numpy as np
import pytest

import oracle
from oracle import gate, online
from attention_forward_gb300 import inputs


def _f(t):
    return t.float().numpy()


CASES = [  # B, H, Sq, Skv, D, causal
    (1, 2, 300, 300, 32, False), (1, 2, 300, 300, 32, True),
    (2, 1, 130, 257, 16, True), (1, 1, 260, 100, 8, True),
    (1, 1, 1, 300, 16, False), (1, 1, 129, 129, 64, True),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("block_n", [128, 64, 1])
def test_online_equals_three_step(case, block_n):
    B, H, Sq, Skv, D, causal = case
    q, k, v = inputs.make_qkv(B, H, Sq, Skv, D, "bf16", 7, qk_mult=4.0)
    q, k, v = _f(q), _f(k), _f(v)
    sc = D ** -0.5
    o_ref, l_ref = oracle.attention(q, k, v, sc, causal)
    o, l = online.online_attention(q, k, v, sc, causal, block_n=block_n)
    assert np.abs(o - o_ref).max() < 1e-12
    fin = np.isfinite(l_ref)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.abs(l[fin] - l_ref[fin]).max() < 1e-12


@pytest.mark.parametrize("nsplit", [1, 2, 3, 7])
def test_split_kv_combine_equals_oracle(nsplit):
    B, H, Sq, Skv, D = 2, 2, 3, 1000, 64
    q, k, v = (_f(t) for t in inputs.make_qkv(B, H, Sq, Skv, D, "bf16", 8))
    sc = D ** -0.5
    o_ref, l_ref = oracle.attention(q, k, v, sc, False)
    bounds = np.linspace(0, Skv, nsplit + 1).astype(int)
    parts = [oracle.attention(q, k[:, :, a:b], v[:, :, a:b], sc, False)
             for a, b in zip(bounds[:-1], bounds[1:])]
    o, l = online.combine_partials([p[0] for p in parts], [p[1] for p in parts])
    assert np.abs(o - o_ref).max() < 1e-12
    assert np.abs(l - l_ref).max() < 1e-12


def test_combine_with_empty_splits():
    o_parts = np.array([[[1.0, 2.0]], [[5.0, 6.0]]])
    lse_parts = np.array([[-np.inf], [0.3]])
    o, l = online.combine_partials(o_parts, lse_parts)
    assert np.array_equal(o, [[5.0, 6.0]]) and abs(l[0] - 0.3) < 1e-15
    o, l = online.combine_partials(o_parts, np.full((2, 1), -np.inf))
    assert np.all(o == 0.0) and np.isneginf(l[0])


GATE_CASES = [  # B, H, S, D, dtype, causal, qk_mult
    (1, 2, 300, 64, "bf16", False, 1.0), (1, 2, 300, 64, "bf16", True, 1.0),
    (1, 2, 300, 64, "fp16", True, 1.0), (1, 2, 300, 64, "bf16", True, 4.0),
    (1, 2, 300, 128, "bf16", False, 4.0),
]


def _gate_inputs(case):
    B, H, S, D, dtype, causal, mult = case
    q, k, v = (_f(t) for t in inputs.make_qkv(B, H, S, S, D, dtype, 9, mult))
    sc = D ** -0.5
    fmt = oracle.FMT_BF16 if dtype == "bf16" else oracle.FMT_F16
    o_ref, l_ref = oracle.attention(q, k, v, sc, causal)
    o_fl, _ = oracle.floor_attention(q, k, v, sc, causal, fmt)
    return q, k, v, sc, causal, dtype, fmt, o_ref, l_ref, o_fl


@pytest.fixture(scope="module")
def gate_inputs():
    return [_gate_inputs(c) for c in GATE_CASES]


def test_gate_admits_rounded_online_softmax(gate_inputs):
    """The algorithm with P and O rounded to the 16-bit format, as the kernel
    does, passes the gate on every case."""
    for q, k, v, sc, causal, dtype, fmt, o_ref, l_ref, o_fl in gate_inputs:
        rnd = lambda x: oracle.round_fmt(x, fmt).astype(np.float64)
        o, l = online.online_attention(q, k, v, sc, causal, p_round=rnd)
        r = gate.check(o, l, o_ref, l_ref, o_fl, dtype)
        assert r.passed, str(r)


@pytest.mark.parametrize("mutation", online.MUTATIONS)
def test_gate_rejects_planted_mistake(gate_inputs, mutation):
    """Every planted mistake fails the gate on at least one case."""
    results = []
    for q, k, v, sc, causal, dtype, fmt, o_ref, l_ref, o_fl in gate_inputs:
        rnd = lambda x: oracle.round_fmt(x, fmt).astype(np.float64)
        with np.errstate(all="ignore"):
            o, l = online.online_attention(q, k, v, sc, causal, p_round=rnd,
                                           mutation=mutation)
        results.append(gate.check(o, l, o_ref, l_ref, o_fl, dtype).passed)
    assert not all(results), f"gate passed mutation {mutation} everywhere"
