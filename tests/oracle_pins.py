"""Pins for the fp64 oracle: facts fixed by mathematics or by an independent
library routine, not by the oracle itself.

Each ``pin_*`` takes a loaded oracle library (``oracle.load(...)``) and raises
AssertionError when the oracle disagrees.  ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle
with planted mistakes and requires that every mutant fails at least one pin.

Definitions pinned (all bottom-right causal):
  s_ij = scale * q_i . k_j, visible j <= i + Skv - Sq when causal,
  O_i = softmax_j(s_ij) V, LSE_i = ln sum_j exp(s_ij).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

RNG = np.random.default_rng(20261202)


def _rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def _mask(Sq, Skv, causal):
    i = np.arange(Sq)[:, None]
    j = np.arange(Skv)[None, :]
    return (j <= i + (Skv - Sq)) if causal else np.ones((Sq, Skv), bool)


def pin_library_sdpa(lib):
    """Torch's CPU scaled_dot_product_attention in float64 (an independent
    library routine) with an explicit bottom-right boolean mask, and
    torch.logsumexp for LSE, on small random problems."""
    cases = [(2, 3, 5, 7, 8, False), (2, 3, 5, 7, 8, True),
             (1, 2, 7, 5, 4, True), (1, 2, 9, 9, 16, True),
             (2, 1, 6, 13, 3, False), (1, 1, 1, 11, 5, True)]
    for B, H, Sq, Skv, D, causal in cases:
        q, k, v = _rand(B, H, Sq, D), _rand(B, H, Skv, D), _rand(B, H, Skv, D)
        scale = 0.37
        o, lse = oracle.attention(q, k, v, scale, causal, nthreads=2, lib=lib)
        m = _mask(Sq, Skv, causal)
        live = m.any(axis=1)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        tm = torch.from_numpy(m)
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=tm, scale=scale).numpy()
        s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
        s = s.masked_fill(~tm, float("-inf"))
        ref_lse = torch.logsumexp(s, dim=-1).numpy()
        assert np.abs(o[:, :, live] - ref[:, :, live]).max() < 1e-12, (B, H, Sq, Skv)
        assert np.abs(lse[:, :, live] - ref_lse[:, :, live]).max() < 1e-12
        assert np.all(o[:, :, ~live] == 0.0)
        assert np.all(np.isneginf(lse[:, :, ~live]))


def pin_q_zero(lib):
    """Q = 0: every visible score is 0, so O_i is the mean of the visible V
    rows and LSE_i = ln(number of visible keys)."""
    for Sq, Skv, causal in [(6, 6, True), (4, 9, True), (5, 7, False)]:
        B, H, D = 2, 2, 5
        q = np.zeros((B, H, Sq, D))
        k, v = _rand(B, H, Skv, D), _rand(B, H, Skv, D)
        o, lse = oracle.attention(q, k, v, 0.5, causal, lib=lib)
        for i in range(Sq):
            n = min(Skv, i + Skv - Sq + 1) if causal else Skv
            assert np.abs(o[:, :, i] - v[:, :, :n].mean(axis=2)).max() < 1e-13
            assert np.abs(lse[:, :, i] - math.log(n)).max() < 1e-13


def pin_causal_row0(lib):
    """Causal with Sq = Skv: row 0 sees only key 0, so O_0 = V_0 and
    LSE_0 = scale * q_0 . k_0."""
    B, H, S, D = 2, 3, 8, 6
    q, k, v = _rand(B, H, S, D), _rand(B, H, S, D), _rand(B, H, S, D)
    o, lse = oracle.attention(q, k, v, 0.3, True, lib=lib)
    assert np.abs(o[:, :, 0] - v[:, :, 0]).max() < 1e-14
    s00 = 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    assert np.abs(lse[:, :, 0] - s00).max() < 1e-13


def pin_dominant_key(lib):
    """A key whose score beats every other by >= 40 takes all the weight:
    O_i = v_pi(i) up to Skv * exp(-40) * max|v|; LSE_i = s_i,pi(i) + O(e^-40)."""
    B, H, S, D = 1, 2, 8, 16
    scale = 0.25
    perm = np.array([3, 0, 7, 1, 6, 2, 5, 4])
    q = np.zeros((B, H, S, D))
    k = np.zeros((B, H, S, D))
    for i in range(S):
        q[:, :, i, perm[i]] = 45.0 / scale
    for j in range(S):
        k[:, :, j, j] = 1.0
    k += _rand(B, H, S, D, scale=1e-3)
    v = _rand(B, H, S, D)
    o, lse = oracle.attention(q, k, v, scale, False, lib=lib)
    for i in range(S):
        assert np.abs(o[:, :, i] - v[:, :, perm[i]]).max() < 1e-12
        s_dom = scale * np.einsum("bhd,bhd->bh", q[:, :, i], k[:, :, perm[i]])
        assert np.abs(lse[:, :, i] - s_dom).max() < 1e-12


def pin_probs(lib):
    """P rows are non-negative, zero at masked keys, sum to 1, and
    O = P V (step 3 uses the step-2 probabilities)."""
    for Sq, Skv, causal in [(7, 7, True), (5, 9, True), (6, 4, False)]:
        D = 5
        q, k, v = _rand(Sq, D), _rand(Skv, D), _rand(Skv, D)
        P = oracle.probs(q, k, 0.6, causal, lib=lib)
        m = _mask(Sq, Skv, causal)
        assert np.all(P >= 0.0)
        assert np.all(P[~m] == 0.0)
        live = m.any(axis=1)
        assert np.abs(P[live].sum(axis=1) - 1.0).max() < 1e-15 * Skv + 1e-15
        o, _ = oracle.attention(q[None, None], k[None, None], v[None, None],
                                0.6, causal, lib=lib)
        assert np.abs(o[0, 0][live] - P[live] @ v).max() < 1e-13


def pin_shift_invariance(lib):
    """Adding c_i to every score of row i leaves O unchanged and shifts LSE by
    c_i.  Realised with one extra feature: q'_i = [q_i, c_i/scale],
    k'_j = [k_j, 1]."""
    B, H, Sq, Skv, D = 1, 2, 6, 9, 4
    scale = 0.7
    q, k, v = _rand(B, H, Sq, D), _rand(B, H, Skv, D), _rand(B, H, Skv, D)
    c = np.linspace(-30.0, 55.0, Sq)
    q2 = np.concatenate([q, np.broadcast_to((c / scale)[None, None, :, None],
                                            (B, H, Sq, 1))], axis=-1)
    k2 = np.concatenate([k, np.ones((B, H, Skv, 1))], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, Skv, 1))], axis=-1)
    for causal in (False, True):
        o1, l1 = oracle.attention(q, k, v, scale, causal, lib=lib)
        o2, l2 = oracle.attention(q2, k2, v2, scale, causal, lib=lib)
        assert np.all(o2[..., D] == 0.0)
        assert np.abs(o1 - o2[..., :D]).max() < 1e-12
        assert np.abs(l2 - (l1 + c)).max() < 1e-11


def pin_single_key_and_two_keys(lib):
    """Skv = 1: O = v_0, LSE = scale q.k_0.  Skv = 2, D = 1: the closed form
    O = (e^s1 v1 + e^s2 v2) / (e^s1 + e^s2), LSE = ln(e^s1 + e^s2)."""
    q, k, v = _rand(1, 1, 3, 4), _rand(1, 1, 1, 4), _rand(1, 1, 1, 4)
    o, lse = oracle.attention(q, k, v, 1.3, False, lib=lib)
    assert np.abs(o[0, 0] - v[0, 0, 0][None]).max() < 1e-15
    assert np.abs(lse[0, 0] - 1.3 * (q[0, 0] @ k[0, 0, 0])).max() < 1e-14
    a, b1, b2, v1, v2, sc = 0.8, 1.5, -0.25, 2.0, -3.0, 0.9
    q = np.array([[[[a]]]])
    k = np.array([[[[b1], [b2]]]])
    v = np.array([[[[v1], [v2]]]])
    o, lse = oracle.attention(q, k, v, sc, False, lib=lib)
    s1, s2 = sc * a * b1, sc * a * b2
    e1, e2 = math.exp(s1), math.exp(s2)
    assert abs(o[0, 0, 0, 0] - (e1 * v1 + e2 * v2) / (e1 + e2)) < 1e-15
    assert abs(lse[0, 0, 0] - math.log(e1 + e2)) < 1e-15


def pin_heads_independent(lib):
    """Each (b, h) uses only its own K/V: a head computed alone matches the
    same head inside a batch; permuting keys (K and V rows together) leaves a
    non-causal output unchanged."""
    B, H, Sq, Skv, D = 2, 3, 5, 6, 4
    q, k, v = _rand(B, H, Sq, D), _rand(B, H, Skv, D), _rand(B, H, Skv, D)
    o, lse = oracle.attention(q, k, v, 0.5, True, lib=lib)
    for b in range(B):
        for h in range(H):
            o1, l1 = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                      v[b:b + 1, h:h + 1], 0.5, True, lib=lib)
            assert np.abs(o1[0, 0] - o[b, h]).max() < 1e-15
            assert np.abs(l1[0, 0] - lse[b, h]).max() < 1e-15
    perm = RNG.permutation(Skv)
    o1, l1 = oracle.attention(q, k, v, 0.5, False, lib=lib)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.5, False,
                              lib=lib)
    assert np.abs(o1 - o2).max() < 1e-13 and np.abs(l1 - l2).max() < 1e-13


def pin_rows_path(lib):
    """The sampled-rows entry gives, row for row, the full-tensor result."""
    B, H, Sq, Skv, D = 2, 2, 7, 7, 3
    q, k, v = _rand(B, H, Sq, D), _rand(B, H, Skv, D), _rand(B, H, Skv, D)
    o, lse = oracle.attention(q, k, v, 0.4, True, lib=lib)
    rows = np.array([0, 27, 13, 6, 7, 20])
    o_r, l_r = oracle.attention(q, k, v, 0.4, True, rows=rows, lib=lib)
    assert np.array_equal(o_r, o.reshape(-1, D)[rows])
    assert np.array_equal(l_r, lse.reshape(-1)[rows])


def pin_fully_masked(lib):
    """Causal with Sq > Skv: rows i < Sq - Skv see no key: O = 0, LSE = -inf;
    row Sq - Skv sees only key 0."""
    B, H, Sq, Skv, D = 1, 1, 6, 3, 4
    q, k, v = _rand(B, H, Sq, D), _rand(B, H, Skv, D), _rand(B, H, Skv, D)
    o, lse = oracle.attention(q, k, v, 0.5, True, lib=lib)
    assert np.all(o[0, 0, :3] == 0.0) and np.all(np.isneginf(lse[0, 0, :3]))
    assert np.abs(o[0, 0, 3] - v[0, 0, 0]).max() < 1e-15


ALL_PINS = [pin_library_sdpa, pin_q_zero, pin_causal_row0, pin_dominant_key,
            pin_probs, pin_shift_invariance, pin_single_key_and_two_keys,
            pin_heads_independent, pin_rows_path, pin_fully_masked]


# ------------------------------------------------------------------ floor
#
# The fp32 same-precision floor (``floor_attention_rows``) sets half of the
# parity bound, so a mistake that inflates its error would loosen the gate.
# Its definition: fp32 scores, fp32 softmax with expf, the normalised P
# rounded to the 16-bit input format, fp32 P.V, O rounded to the format
# (round to nearest even); LSE = m + ln l in fp32.

_TORCH_FMT = {oracle.FMT_BF16: torch.bfloat16, oracle.FMT_F16: torch.float16}


def _to_fmt(x, fmt):
    """Round to the 16-bit format through torch's cast (not the oracle's)."""
    return torch.as_tensor(np.asarray(x, np.float32)).to(_TORCH_FMT[fmt]).float().numpy()


def _fmt_inputs(shape, fmt, scale=1.0):
    return _to_fmt(RNG.standard_normal(shape) * scale, fmt)


def _fmt_ulp(x, fmt):
    """Spacing of the 16-bit format at |x| (normal range)."""
    mant, emin = (7, -126) if fmt == oracle.FMT_BF16 else (10, -14)
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 2.0 ** (e - mant)


def pin_floor_library_path(lib):
    """The floor against torch's own fp32 CPU routines on the same 16-bit
    inputs: fp32 matmul for the scores, torch.softmax, P cast to the format,
    fp32 matmul with V, O cast to the format, torch.logsumexp for LSE.  The
    two differ only in fp32 summation order, which moves O by at most one
    unit of the format and almost never across a rounding boundary; LSE
    agrees to fp32 rounding."""
    cases = [(1, 2, 96, 160, 64, False, oracle.FMT_BF16, 1.0),
             (1, 2, 96, 160, 64, True, oracle.FMT_BF16, 1.0),
             (1, 2, 80, 80, 32, True, oracle.FMT_F16, 1.0),
             (1, 1, 64, 200, 16, False, oracle.FMT_F16, 3.0)]
    for B, H, Sq, Skv, D, causal, fmt, mult in cases:
        q = _fmt_inputs((B, H, Sq, D), fmt, mult)
        k = _fmt_inputs((B, H, Skv, D), fmt, mult)
        v = _fmt_inputs((B, H, Skv, D), fmt)
        scale = float(np.float32(D ** -0.5))
        of, lf = oracle.floor_attention(q, k, v, scale, causal, fmt, nthreads=2,
                                        lib=lib)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        s = torch.matmul(tq, tk.transpose(-1, -2)) * scale
        m = torch.from_numpy(_mask(Sq, Skv, causal))
        s = s.masked_fill(~m, float("-inf"))
        live = m.any(dim=1).numpy()
        p = torch.softmax(s, dim=-1).to(_TORCH_FMT[fmt]).float()
        o = torch.matmul(p, tv).to(_TORCH_FMT[fmt]).float().numpy()
        lse = torch.logsumexp(s, dim=-1).numpy()
        of_l, o_l = of[:, :, live], o[:, :, live]
        diff = np.abs(of_l - o_l)
        # a P value next to a rounding boundary of the format may round the
        # other way in torch (its softmax multiplies by 1/l), which moves
        # that row's O by a unit of P: allow it on a few rows
        rows_off = np.any(diff > _fmt_ulp(o_l, fmt) * 1.0001, axis=-1)
        assert np.mean(rows_off) <= 0.03, (Sq, Skv, causal, fmt, np.mean(rows_off))
        assert np.mean(diff == 0.0) >= 0.99, np.mean(diff == 0.0)
        assert np.abs(lf[:, :, live] - lse[:, :, live]).max() < 4e-6


def pin_floor_q_zero_closed_form(lib):
    """Q = 0: every visible score is exactly 0, expf(0) = 1, l = n, so the
    floor's P is 1/n rounded to fp32 and then to the format, and with small
    integer V every fp32 sum is exact: O_i = fmt(P * sum of the visible V
    rows), LSE_i = ln n."""
    for fmt in (oracle.FMT_BF16, oracle.FMT_F16):
        Sq = Skv = 40
        D = 8
        q = np.zeros((1, 1, Sq, D), np.float32)
        k = _fmt_inputs((1, 1, Skv, D), fmt)
        v = RNG.integers(-8, 9, size=(1, 1, Skv, D)).astype(np.float32)
        of, lf = oracle.floor_attention(q, k, v, 0.125, True, fmt, lib=lib)
        for i in range(Sq):
            n = i + 1
            p = float(_to_fmt(np.float32(1.0) / np.float32(n), fmt))
            expect = _to_fmt(p * v[0, 0, :n].astype(np.float64).sum(axis=0), fmt)
            assert np.array_equal(of[0, 0, i], expect), (fmt, i)
            assert abs(float(lf[0, 0, i]) - math.log(n)) < 2e-6


def pin_floor_single_key_exact(lib):
    """One visible key (causal row 0): P = 1 exactly, so O_0 = V_0 exactly
    and LSE_0 = the fp32 score."""
    for fmt in (oracle.FMT_BF16, oracle.FMT_F16):
        q = _fmt_inputs((1, 1, 4, 64), fmt)
        k = _fmt_inputs((1, 1, 4, 64), fmt)
        v = _fmt_inputs((1, 1, 4, 64), fmt)
        of, lf = oracle.floor_attention(q, k, v, 0.125, True, fmt, lib=lib)
        assert np.array_equal(of[0, 0, 0], v[0, 0, 0])
        s00 = 0.125 * float(q[0, 0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64))
        assert abs(float(lf[0, 0, 0]) - s00) < 1e-5


def pin_floor_output_on_grid(lib):
    """Every floor output is a value of the 16-bit format (the output is
    rounded once at the end)."""
    for fmt in (oracle.FMT_BF16, oracle.FMT_F16):
        q, k, v = (_fmt_inputs((1, 2, 50, 32), fmt) for _ in range(3))
        of, _ = oracle.floor_attention(q, k, v, 32 ** -0.5, False, fmt, lib=lib)
        assert np.array_equal(of, _to_fmt(of, fmt))


def pin_floor_within_oracle_rounding(lib):
    """Against the fp64 oracle the floor errs by the 16-bit rounding of O and
    P: a few units of the format, and not zero (it does round)."""
    for fmt, u in ((oracle.FMT_BF16, 2.0 ** -8), (oracle.FMT_F16, 2.0 ** -11)):
        q, k, v = (_fmt_inputs((1, 2, 120, 64), fmt) for _ in range(3))
        for causal in (False, True):
            o, lse = oracle.attention(q, k, v, 0.125, causal, lib=lib)
            of, lf = oracle.floor_attention(q, k, v, 0.125, causal, fmt, lib=lib)
            err = np.abs(of - o).max()
            assert 0.0 < err < 4 * u * np.abs(v).max()
            assert np.abs(lf - lse).max() < 1e-4


FLOOR_PINS = [pin_floor_library_path, pin_floor_q_zero_closed_form,
              pin_floor_single_key_exact, pin_floor_output_on_grid,
              pin_floor_within_oracle_rounding]
