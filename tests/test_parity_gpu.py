"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle,
on the workloads of the build and on edge cases.  Gate: oracle/gate.py."""
import numpy as np
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check, run_and_check, run_kernel, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _assert(r):
    assert r.passed, str(r)


def test_pr1():
    w = inputs.PR1
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed))


@pytest.mark.parametrize("w", [inputs.C2, inputs.C2_CAUSAL, inputs.C2_X4,
                               inputs.C2_X4_CAUSAL], ids=lambda w: w.name)
def test_c2_all_rows(w):
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal,
                          w.seed, w.qk_mult))


EDGE = [  # B, H, Sq, Skv, D, dtype, causal
    (1, 1, 2, 2, 64, "bf16", False), (1, 1, 2, 2, 128, "fp16", True),
    (1, 1, 7, 7, 128, "bf16", True), (2, 3, 127, 127, 64, "fp16", False),
    (1, 2, 128, 128, 128, "bf16", True), (1, 2, 129, 129, 128, "bf16", True),
    (1, 1, 255, 255, 64, "bf16", True), (1, 1, 256, 256, 128, "fp16", True),
    (1, 1, 257, 257, 128, "bf16", False), (2, 2, 300, 300, 64, "bf16", True),
    (1, 2, 1000, 1000, 128, "fp16", True), (1, 1, 100, 300, 128, "bf16", True),
    (1, 1, 100, 300, 64, "fp16", False), (1, 1, 300, 100, 128, "bf16", True),
    (1, 1, 300, 100, 64, "bf16", False), (1, 1, 513, 1, 128, "bf16", False),
    (1, 1, 600, 129, 128, "fp16", True), (3, 1, 384, 640, 64, "bf16", True),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "x".join(map(str, c)))
def test_edge_shapes(case):
    B, H, Sq, Skv, D, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, D, dt, causal, 11, qk_mult=2.0))


# More work items than SMs, so every persistent CTA takes several in turn:
# items without a visible key (causal, Sq > Skv) between others, stages with
# no key tile, many short ragged items, LPT order.
PERSISTENT = [  # B, H, Sq, Skv, D, dtype, causal
    (1, 64, 1024, 128, 128, "bf16", True),
    (4, 48, 600, 129, 128, "bf16", True),
    (8, 32, 300, 300, 64, "fp16", True),
    (8, 32, 300, 300, 128, "bf16", False),
]


@pytest.mark.parametrize("case", PERSISTENT, ids=lambda c: "x".join(map(str, c)))
def test_persistent_item_sequences(case):
    B, H, Sq, Skv, D, dt, causal = case
    _assert(run_and_check(B, H, Sq, Skv, D, dt, causal, 13))


def test_scheduler_slots_wrap_around():
    """1100 launches, more than the 1024 scheduler slots: every launch still
    claims every item (outputs cleared before every 100th launch must come
    back bit for bit)."""
    q, k, v = inputs.make_qkv(4, 64, 512, 512, 128, "bf16", 3)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    ref, lref = fa.fa_fwd(dq, dk, dv, causal=True)
    o, lse = torch.empty_like(ref), torch.empty_like(lref)
    for i in range(1100):
        if i % 100 == 99:
            o.zero_()
            lse.fill_(float("nan"))
        fa.fa_fwd(dq, dk, dv, causal=True, out=o, lse=lse)
        if i % 100 == 99:
            torch.cuda.synchronize()
            assert torch.equal(o, ref) and torch.equal(lse, lref), i
    assert fa.fa_get_device_status() == fa.FA_OK


def test_headline_sampled_rows():
    """B4 H16 S4096 D128 bf16 non-causal at full size, in the launch the bench
    times (fa_fwd, default options); >= 512 sampled rows covering every head."""
    w = inputs.HEADLINE
    rows = rows_at_least(w, seed=1)
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal,
                          w.seed, rows=rows))


def rows_at_least(w, n=512, seed=0):
    """At least n sampled rows of a large workload: tile-edge, first and last
    rows of every head plus random rows, spread so that every head gets its
    share."""
    per_head = max(8, 2 * -(-n // (w.B * w.H)))
    rows = sample_rows(w.B, w.H, w.Sq, per_head=per_head, extra=256, seed=seed)
    assert rows.size >= n and np.unique(rows // w.Sq).size == w.B * w.H
    return rows


@pytest.mark.parametrize("w", [inputs.LONG16K, inputs.LONG32K],
                         ids=lambda w: w.name)
def test_long_causal_sampled_rows(w):
    """Both long causal workloads at full size, >= 512 sampled rows."""
    rows = rows_at_least(w, seed=2)
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal,
                          w.seed, rows=rows))


@pytest.mark.parametrize("w", [w for w in inputs.SWEEP if w.Sq <= 2048],
                         ids=lambda w: w.name)
def test_sweep_all_rows(w):
    """The B*S = 16384 sweep up to S = 2048: every output row."""
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal, w.seed))


@pytest.mark.parametrize("w", [w for w in inputs.SWEEP if w.Sq > 2048],
                         ids=lambda w: w.name)
def test_sweep_sampled_rows(w):
    """The sweep from S = 4096 on: >= 512 sampled rows covering every head."""
    rows = rows_at_least(w, seed=3)
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal,
                          w.seed, rows=rows))


def test_decode_all_rows():
    """Sq=1, Skv=8192, B32 H32 D128 bf16: every output row, the default
    split count (the bench's launch)."""
    w = inputs.DECODE
    _assert(run_and_check(w.B, w.H, w.Sq, w.Skv, w.D, w.dtype, w.causal,
                          w.seed))


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7])
@pytest.mark.parametrize("D,dt,Skv", [(128, "bf16", 1000), (64, "fp16", 513),
                                      (128, "fp16", 64), (64, "bf16", 3)])
def test_decode_splits(num_splits, D, dt, Skv):
    q, k, v = inputs.make_qkv(2, 5, 1, Skv, D, dt, 21, 3.0)
    ws_bytes = fa.fa_workspace_bytes(2, 5, 1, Skv, D, num_splits)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    o, lse = run_kernel(q, k, v, False, num_splits=num_splits, workspace=ws)
    _assert(check(q, k, v, o, lse, False, dt))


PREFILL_SPLITS = [  # B, H, Sq, Skv, D, dtype, causal, num_splits
    (2, 3, 300, 1000, 128, "bf16", True, 2),
    (2, 3, 300, 1000, 128, "bf16", False, 3),
    (1, 2, 700, 2048, 64, "fp16", True, 5),
    (1, 1, 600, 300, 128, "bf16", True, 3),   # some ranges see no key of a row
    (2, 2, 257, 129, 64, "bf16", False, 2),
]


@pytest.mark.parametrize("case", PREFILL_SPLITS, ids=lambda c: "x".join(map(str, c)))
def test_prefill_key_splits(case):
    """Prefill with the keys split into ranges (fp32 partials in the caller's
    workspace, merged by the combine kernel)."""
    B, H, Sq, Skv, D, dt, causal, n = case
    q, k, v = inputs.make_qkv(B, H, Sq, Skv, D, dt, 17, 2.0)
    need = fa.fa_workspace_bytes(B, H, Sq, Skv, D, n)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, lse = run_kernel(q, k, v, causal, num_splits=n, workspace=ws)
    _assert(check(q, k, v, o, lse, causal, dt))
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        run_kernel(q, k, v, causal, num_splits=n, workspace=small)
    assert e.value.status == fa.FA_ERR_WORKSPACE


def test_prefill_few_items_long_keys():
    """A short query block over a long context (8 items on the whole GPU):
    fa_fwd splits the keys by itself."""
    assert fa.fa_workspace_bytes(1, 8, 256, 16384, 128) > 0
    _assert(run_and_check(1, 8, 256, 16384, 128, "bf16", True, 19))


@pytest.mark.parametrize("num_splits", [1, 3])
def test_repeat_lpt_and_rescale_switches_are_bitwise_identical(num_splits):
    q, k, v = inputs.make_qkv(2, 4, 1000, 1000, 128, "bf16", 5, 4.0)
    need = fa.fa_workspace_bytes(2, 4, 1000, 1000, 128, num_splits)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    kw = dict(num_splits=num_splits, workspace=ws)
    o1, l1 = run_kernel(q, k, v, True, **kw)
    o2, l2 = run_kernel(q, k, v, True, **kw)
    o3, l3 = run_kernel(q, k, v, True, flags=fa.FA_FLAG_NO_LPT, **kw)
    o4, l4 = run_kernel(q, k, v, True, flags=fa.FA_FLAG_ALWAYS_RESCALE, **kw)
    for o, l in ((o2, l2), (o3, l3), (o4, l4)):
        assert torch.equal(o, o1) and torch.equal(l, l1)


@pytest.mark.parametrize("w", [inputs.C2_X4, inputs.C2_X4_CAUSAL, inputs.PR1],
                         ids=lambda w: w.name)
def test_exact_running_max_mode(w):
    """FA_FLAG_EXACT_MAX (rescale whenever the row max grows) passes the gate
    too, and switching the rescale off when alpha == 1 changes no bit."""
    q, k, v = w.make()
    o1, l1 = run_kernel(q, k, v, w.causal, flags=fa.FA_FLAG_EXACT_MAX)
    _assert(check(q, k, v, o1, l1, w.causal, w.dtype))
    o2, l2 = run_kernel(q, k, v, w.causal,
                        flags=fa.FA_FLAG_EXACT_MAX | fa.FA_FLAG_ALWAYS_RESCALE)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_concurrent_streams_bitwise_identical():
    q, k, v = inputs.make_qkv(2, 8, 1024, 1024, 128, "bf16", 6)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    ref, lref = fa.fa_fwd(dq, dk, dv, causal=True)
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = []
    for s in streams:
        with torch.cuda.stream(s):
            outs.append(fa.fa_fwd(dq, dk, dv, causal=True, stream=s))
    torch.cuda.synchronize()
    for o, l in outs:
        assert torch.equal(o, ref) and torch.equal(l, lref)


def test_host_buffers_path_matches_device_path():
    for (Sq, Skv, causal) in ((300, 300, True), (1, 700, False)):
        q, k, v = inputs.make_qkv(2, 3, Sq, Skv, 128, "bf16", 7)
        o_d, l_d = run_kernel(q, k, v, causal)
        pin = [t.pin_memory() for t in (q, k, v)]
        staging = torch.empty(fa.fa_host_staging_bytes(2, 3, Sq, Skv, 128),
                              dtype=torch.uint8, device="cuda")
        o_h, l_h = fa.fa_fwd_host(*pin, staging, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


def test_watchdog_reports_timeout_and_context_survives():
    """The test hook withholds one K/V tile: the consumers' bounded waits run
    out, the kernel stops and reports FA_ERR_TIMEOUT, and the next call on the
    same context is correct."""
    q, k, v = inputs.make_qkv(1, 2, 256, 512, 128, "bf16", 8)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_set_watchdog_ns(20_000_000)  # 20 ms
    try:
        fa.fa_fwd_ex(dq, dk, dv, flags=fa.FA_FLAG_TEST_STALL)
        assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
        assert fa.fa_get_device_status() == fa.FA_OK  # cleared
    finally:
        fa.fa_set_watchdog_ns(0)
    o, lse = run_kernel(q, k, v, False)
    _assert(check(q, k, v, o, lse, False, "bf16"))


@pytest.mark.parametrize("w", [inputs.C2_X4, inputs.C2_X4_CAUSAL],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("kflag", [fa.FA_FLAG_SINGLE_CTA, fa.FA_FLAG_PAIR],
                         ids=["single", "pair"])
def test_correction_warpgroup_form_all_rows(w, kflag):
    """The correction-warpgroup form against the oracle on every row of the
    x4 workload (scores four times larger: the reference max moves), in
    exact-max mode so that most tiles go through the correction warps, and
    bitwise equal to the merged form."""
    q, k, v = w.make()
    f = kflag | fa.FA_FLAG_EXACT_MAX
    o1, l1 = run_kernel(q, k, v, w.causal, flags=f | fa.FA_FLAG_CORRECTION_WG)
    _assert(check(q, k, v, o1, l1, w.causal, w.dtype))
    o2, l2 = run_kernel(q, k, v, w.causal, flags=f)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_correction_warpgroup_watchdog():
    """A withheld K/V tile with the correction warps polling: the watchdog
    still ends every role and reports FA_ERR_TIMEOUT; the next call works."""
    q, k, v = inputs.make_qkv(1, 2, 256, 512, 128, "bf16", 8)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    assert fa.fa_get_device_status() == fa.FA_OK
    fa.fa_set_watchdog_ns(20_000_000)
    try:
        for kflag in (fa.FA_FLAG_SINGLE_CTA, fa.FA_FLAG_PAIR):
            fa.fa_fwd_ex(dq, dk, dv, flags=kflag | fa.FA_FLAG_CORRECTION_WG |
                         fa.FA_FLAG_TEST_STALL)
            assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
    finally:
        fa.fa_set_watchdog_ns(0)
    o, lse = run_kernel(q, k, v, False, flags=fa.FA_FLAG_CORRECTION_WG)
    _assert(check(q, k, v, o, lse, False, "bf16"))
