"""Numerically demanding inputs through the C ABI, on the single-CTA kernel
(D 128 and 64) and on CTA pairs, against the fp64 oracle with the gate of
oracle/gate.py: a sharp softmax (scale 1, so that the reference max moves and
the rescale path runs), a nearly flat one (scale 1e-3: O close to the mean of
V over every key), and keys whose scores grow along the sequence, so that the
row max rises from tile to tile (default threshold and exact-max mode)."""
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check, run_kernel

pytestmark = pytest.mark.gpu

KERNELS = [  # name, D, flags
    ("single_d128", 128, fa.FA_FLAG_SINGLE_CTA),
    ("single_d64", 64, fa.FA_FLAG_SINGLE_CTA),
    ("pair", 128, fa.FA_FLAG_PAIR),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k[0])
@pytest.mark.parametrize("scale", [1.0, 1e-3], ids=["sharp", "flat"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_extreme_scales(kernel, scale, causal):
    """V is scaled by 1/4 (exactly, in bf16): at scale 1 each output row is
    close to a single V row, and with N(0, 1) values the bf16 rounding of P
    and O alone puts the fp32 same-precision floor at 2.3e-2 (D = 64), above
    the gate's absolute bf16 cap of 2e-2 that the configured workloads were
    set against."""
    _, D, flags = kernel
    q, k, v = inputs.make_qkv(1, 4, 1500, 1500, D, "bf16", 51)
    v = v * 0.25
    o, lse = run_kernel(q, k, v, causal, flags=flags, scale=scale)
    r = check(q, k, v, o, lse, causal, "bf16", scale=scale)
    assert r.passed, str(r)


def _ramped(D, dt, seed):
    """Seeded inputs with K scaled by 1 + 3j/Skv along the keys (then rounded
    to the 16-bit format): later keys score higher, so each row's max keeps
    rising across key tiles."""
    q, k, v = inputs.make_qkv(1, 4, 1100, 1100, D, dt, seed, qk_mult=2.0)
    ramp = 1.0 + 3.0 * torch.arange(k.shape[2], dtype=torch.float32) / k.shape[2]
    k = (k.float() * ramp[None, None, :, None]).to(k.dtype)
    return q, k, v


@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k[0])
@pytest.mark.parametrize("exact", [False, True], ids=["tau8", "exact_max"])
def test_row_max_rising_across_tiles(kernel, exact):
    _, D, flags = kernel
    q, k, v = _ramped(D, "fp16", 52)
    f = flags | (fa.FA_FLAG_EXACT_MAX if exact else 0)
    o, lse = run_kernel(q, k, v, False, flags=f)
    r = check(q, k, v, o, lse, False, "fp16")
    assert r.passed, str(r)
    # rescaling on every tile changes no bit
    o2, l2 = run_kernel(q, k, v, False, flags=f | fa.FA_FLAG_ALWAYS_RESCALE)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("scale", [1.0, 1e-3], ids=["sharp", "flat"])
@pytest.mark.parametrize("shape", [(2, 4, 1, 5000), (1, 2, 256, 8192)], ids=["decode", "split_prefill"])
def test_extreme_scales_through_key_splits(shape, scale, D):
    """Decode and a prefill with few query tiles split their keys and merge
    the ranges' (O, LSE) by LSE weights: a sharp softmax puts nearly all the
    weight in one range.  V scaled by 1/4 as in test_extreme_scales."""
    B, H, Sq, Skv = shape
    assert fa.fa_workspace_bytes(B, H, Sq, Skv, D) > 0  # the library splits these
    q, k, v = inputs.make_qkv(B, H, Sq, Skv, D, "bf16", 53)
    v = v * 0.25
    o, lse = run_kernel(q, k, v, False, scale=scale)
    r = check(q, k, v, o, lse, False, "bf16", scale=scale)
    assert r.passed, str(r)


def test_ex2_special_values_on_the_device():
    """The exponential every kernel's softmax uses (ex2.approx.ftz.f32, run
    through fa_ex2_approx): 2^-inf = +0 (masked keys), 2^0 = 1 (the row max),
    exact powers of two, results below the normal range flushed to +0,
    +inf and NaN propagated ("The FA5090 Optimization Journey", section 2.6,
    asserts the first two on the device)."""
    import math
    x = torch.tensor([-math.inf, 0.0, -0.0, 1.0, -1.0, 8.0, -8.0, 100.0, -126.0,
                      -127.5, -200.0, math.inf, math.nan], device="cuda")
    y = fa.fa_ex2_approx(x).cpu()
    torch.cuda.synchronize()
    bits = y.view(torch.int32)
    assert bits[0].item() == 0          # +0, not -0
    assert y[1].item() == 1.0 and y[2].item() == 1.0
    assert y[3].item() == 2.0 and y[4].item() == 0.5
    assert y[5].item() == 256.0 and y[6].item() == 2.0 ** -8
    assert y[7].item() == 2.0 ** 100
    assert y[8].item() == 2.0 ** -126
    assert bits[9].item() == 0 and bits[10].item() == 0   # flushed to +0
    assert math.isinf(y[11].item()) and y[11].item() > 0
    assert math.isnan(y[12].item())


def test_ex2_accuracy_over_the_softmax_range():
    """Relative error of 2^x against fp64 over the arguments the softmax
    sees (x <= 0 after the max is subtracted, and a little above 0 under the
    lazy-rescale threshold): within 2^-20, far below the 16-bit rounding of
    P."""
    import numpy as np
    g = torch.Generator().manual_seed(7)
    x = torch.cat([torch.rand(200000, generator=g) * -120.0,
                   torch.rand(50000, generator=g) * 8.0 - 4.0])
    y = fa.fa_ex2_approx(x.cuda()).cpu().double().numpy()
    ref = np.exp2(x.double().numpy())
    rel = np.abs(y - ref) / ref
    assert rel.max() <= 2.0 ** -20, rel.max()


@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k[0])
def test_special_values_through_the_hot_path(kernel):
    """Causal rows with exactly one visible key: its score is the row max,
    so p = 2^0 = 1, every other key is masked to -inf and gives p = 2^-inf
    = 0, l = 1: the output row is that V row bit for bit, and LSE is the
    scaled score.  Rows with no visible key (Sq > Skv, bottom-right causal)
    give O = 0 and LSE = -inf."""
    _, D, flags = kernel
    Sq, Skv = 700, 600   # rows 0..99 see no key, row 100 sees key 0 only
    q, k, v = inputs.make_qkv(1, 3, Sq, Skv, D, "bf16", 61)
    o, lse = run_kernel(q, k, v, True, flags=flags)
    o, lse = o.cpu(), lse.cpu()
    assert torch.all(o[:, :, :100] == 0) and torch.all(torch.isneginf(lse[:, :, :100]))
    assert torch.equal(o[:, :, 100], v[:, :, 0])
    s00 = (q[:, :, 100].double() * k[:, :, 0].double()).sum(-1) * D ** -0.5
    assert (lse[:, :, 100].double() - s00).abs().max().item() < 1e-5


@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k[0])
@pytest.mark.parametrize("exact", [False, True], ids=["tau8", "exact_max"])
@pytest.mark.parametrize("always", [False, True], ids=["on_change", "every_tile"])
def test_correction_warpgroup_form_matches_merged_form(kernel, exact, always):
    """FA_FLAG_CORRECTION_WG: a dedicated correction warp rescales O in
    tensor memory for the tiles whose rows moved their max (the softmax warps
    hand those tiles over).  It multiplies each element of O by the same
    alpha as the merged form, so the outputs are the same bits; with the
    exact running max and on every tile the hand-over happens on most tiles.
    Rows whose max keeps rising (the ramped keys) and x4 scores."""
    _, D, flags = kernel
    q, k, v = _ramped(D, "bf16", 54)
    f = flags | (fa.FA_FLAG_EXACT_MAX if exact else 0) | \
        (fa.FA_FLAG_ALWAYS_RESCALE if always else 0)
    o1, l1 = run_kernel(q, k, v, True, flags=f)
    o2, l2 = run_kernel(q, k, v, True, flags=f | fa.FA_FLAG_CORRECTION_WG)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    r = check(q, k, v, o2, l2, True, "bf16")
    assert r.passed, str(r)
