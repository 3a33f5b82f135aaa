"""The C-ABI calls captured into CUDA graphs (torch.cuda.CUDAGraph): replays
give the results of direct calls (bitwise where the same kernel and key split
run), a captured fa_fwd runs unsplit without a library workspace, and graph
replays overlap direct launches that rotate through the scheduler's slots.
Gate: oracle/gate.py."""
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _dev(B, H, Sq, Skv, D, dt, seed):
    q, k, v = inputs.make_qkv(B, H, Sq, Skv, D, dt, seed)
    return (q, k, v), tuple(t.cuda() for t in (q, k, v))


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _replay(g, o, lse, times=3):
    got = []
    for _ in range(times):
        o.zero_()
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got.append((o.clone(), lse.clone()))
    assert fa.fa_get_device_status() == fa.FA_OK
    return got


SAME = [  # B, H, Sq, Skv, D, dtype, causal: no key split, direct or captured
    (4, 8, 2048, 2048, 128, "bf16", False),   # CTA pairs
    (2, 32, 1024, 512, 128, "bf16", True),    # single CTAs, more items than SMs
    (2, 4, 700, 700, 64, "fp16", True),
]


@pytest.mark.parametrize("case", SAME, ids=lambda c: "x".join(map(str, c)))
def test_replays_equal_direct_calls_bitwise(case):
    B, H, Sq, Skv, D, dt, causal = case
    _, (q, k, v) = _dev(B, H, Sq, Skv, D, dt, 41)
    ref, lref = fa.fa_fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    o, lse = torch.empty_like(ref), torch.empty_like(lref)
    g = _capture(lambda: fa.fa_fwd(q, k, v, causal=causal, out=o, lse=lse))
    for go, gl in _replay(g, o, lse):
        assert torch.equal(go, ref) and torch.equal(gl, lref)


@pytest.mark.parametrize("case", [(1, 2, 256, 4096, 128, "bf16", False),
                                  (2, 4, 1, 700, 128, "bf16", False)],
                         ids=["prefill_split", "decode"])
def test_captured_fa_fwd_runs_unsplit_and_passes_the_gate(case):
    """Shapes that fa_fwd splits directly (few query tiles; decode) run
    unsplit inside a capture, where no library workspace is used."""
    B, H, Sq, Skv, D, dt, causal = case
    assert fa.fa_workspace_bytes(B, H, Sq, Skv, D) > 0
    (qc, kc, vc), (q, k, v) = _dev(B, H, Sq, Skv, D, dt, 42)
    # the same computation called directly, unsplit (also loads its kernel
    # before the capture)
    o1, l1 = fa.fa_fwd_ex(q, k, v, causal=causal, num_splits=1)
    torch.cuda.synchronize()
    o, lse = torch.empty_like(o1), torch.empty_like(l1)
    g = _capture(lambda: fa.fa_fwd(q, k, v, causal=causal, out=o, lse=lse))
    got = _replay(g, o, lse)
    for go, gl in got:
        assert torch.equal(go, o1) and torch.equal(gl, l1)
    r = check(qc, kc, vc, got[0][0], got[0][1], causal, dt)
    assert r.passed, str(r)


def test_captured_fa_fwd_ex_keeps_the_split_with_a_caller_workspace():
    B, H, Sq, Skv, D, dt = 1, 2, 256, 4096, 128, "bf16"
    _, (q, k, v) = _dev(B, H, Sq, Skv, D, dt, 43)
    ws = torch.empty(fa.fa_workspace_bytes(B, H, Sq, Skv, D), dtype=torch.uint8, device="cuda")
    ref, lref = fa.fa_fwd_ex(q, k, v, workspace=ws)
    torch.cuda.synchronize()
    o, lse = torch.empty_like(ref), torch.empty_like(lref)
    g = _capture(lambda: fa.fa_fwd_ex(q, k, v, workspace=ws, out=o, lse=lse))
    for go, gl in _replay(g, o, lse):
        assert torch.equal(go, ref) and torch.equal(gl, lref)


def test_captured_host_buffer_call():
    B, H, S, D, dt = 1, 4, 640, 128, "bf16"
    (qc, kc, vc), (q, k, v) = _dev(B, H, S, S, D, dt, 44)
    ref, lref = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    qh, kh, vh = (t.pin_memory() for t in (qc, kc, vc))
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    staging = torch.empty(fa.fa_host_staging_bytes(B, H, S, S, D), dtype=torch.uint8, device="cuda")
    g = _capture(lambda: fa.fa_fwd_host(qh, kh, vh, staging, causal=True, out_h=oh, lse_h=lh))
    for _ in range(2):
        oh.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(oh, ref.cpu()) and torch.equal(lh, lref.cpu())


def test_replays_overlap_direct_launches_through_the_slot_rotation():
    """A captured prefill keeps its scheduler slot; 1100 direct launches on
    another stream rotate through all of theirs while the graph replays."""
    _, (q, k, v) = _dev(2, 32, 1024, 512, 128, "bf16", 45)
    _, (q2, k2, v2) = _dev(2, 32, 768, 384, 128, "bf16", 46)
    ref, lref = fa.fa_fwd(q, k, v, causal=True)
    ref2, lref2 = fa.fa_fwd(q2, k2, v2, causal=True)
    torch.cuda.synchronize()
    o, lse = torch.empty_like(ref), torch.empty_like(lref)
    g = _capture(lambda: fa.fa_fwd(q, k, v, causal=True, out=o, lse=lse))
    o2, l2 = torch.empty_like(ref2), torch.empty_like(lref2)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for i in range(1100):
        with torch.cuda.stream(sb):
            fa.fa_fwd(q2, k2, v2, causal=True, out=o2, lse=l2)
        if i % 25 == 0:
            with torch.cuda.stream(sa):
                o.zero_()
                g.replay()
        if i % 100 == 99:
            torch.cuda.synchronize()
            assert torch.equal(o, ref) and torch.equal(lse, lref), i
            assert torch.equal(o2, ref2) and torch.equal(l2, lref2), i
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
