"""FA_FLAG_OVERLAP_PREVIOUS: the prefill kernel may start while the previous
grid on the stream is still running (programmatic dependent launch); it
reads Q, K, V early and waits for that grid before its first write.  The
results must be those of plain calls, and every write must land after the
previous grid's writes to the same buffers."""
import pytest
import torch

from attention_forward_gb300 import fa, inputs
from parity import check

pytestmark = pytest.mark.gpu

OV = fa.FA_FLAG_OVERLAP_PREVIOUS
KERNELS = [  # id, B, H, S, D, causal, flags
    ("pair", 4, 16, 2048, 128, False, fa.FA_FLAG_PAIR),
    ("single_causal", 2, 16, 2048, 128, True, fa.FA_FLAG_SINGLE_CTA),
    ("single_d64", 2, 16, 2048, 64, False, 0),
    ("pair_causal", 1, 16, 8192, 128, True, 0),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _dev(*ts):
    return tuple(t.cuda() for t in ts)


@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k[0])
def test_back_to_back_calls_match_plain_calls(kernel):
    _, B, H, S, D, causal, flags = kernel
    q, k, v = _dev(*inputs.make_qkv(B, H, S, S, D, "bf16", 81))
    ref_o, ref_l = fa.fa_fwd_ex(q, k, v, causal=causal, flags=flags)
    o, lse = torch.empty_like(ref_o), torch.empty_like(ref_l)
    for _ in range(20):
        fa.fa_fwd_ex(q, k, v, causal=causal, flags=flags | OV, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k[0])
def test_writes_land_after_the_previous_grid(kernel):
    """Alternating inputs into one output buffer: each overlapped call's
    results must replace the previous call's, so the buffer ends with the
    last call's results, bit for bit."""
    _, B, H, S, D, causal, flags = kernel
    xa = _dev(*inputs.make_qkv(B, H, S, S, D, "bf16", 82))
    xb = _dev(*inputs.make_qkv(B, H, S, S, D, "bf16", 83, 2.0))
    ra = fa.fa_fwd_ex(*xa, causal=causal, flags=flags)
    rb = fa.fa_fwd_ex(*xb, causal=causal, flags=flags)
    o, lse = torch.empty_like(ra[0]), torch.empty_like(ra[1])
    for i in range(31):
        x = xa if i % 2 == 0 else xb
        fa.fa_fwd_ex(*x, causal=causal, flags=flags | OV, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, ra[0]) and torch.equal(lse, ra[1])
    fa.fa_fwd_ex(*xb, causal=causal, flags=flags | OV, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, rb[0]) and torch.equal(lse, rb[1])


def test_after_another_kernel_writing_the_output():
    """A foreign kernel (a fill) writes the output buffers just before an
    overlapped call: the call's results must come after it."""
    q, k, v = inputs.make_qkv(4, 16, 2048, 2048, 128, "bf16", 84)
    dq, dk, dv = _dev(q, k, v)
    ref_o, ref_l = fa.fa_fwd(dq, dk, dv)
    o, lse = torch.empty_like(ref_o), torch.empty_like(ref_l)
    for _ in range(10):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        fa.fa_fwd_ex(dq, dk, dv, flags=OV, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_split_keys_with_overlap():
    """A prefill with split keys (partials in a workspace, then the combine
    kernel) launched overlapped, back to back: the partials are written
    only after the previous grid, which may still be the previous call's
    combine reading them."""
    B, H, Sq, Skv, D = 1, 2, 256, 8192, 128
    q, k, v = inputs.make_qkv(B, H, Sq, Skv, D, "bf16", 85)
    dq, dk, dv = _dev(q, k, v)
    need = fa.fa_workspace_bytes(B, H, Sq, Skv, D)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for _ in range(10):
        o, lse = fa.fa_fwd_ex(dq, dk, dv, causal=True, flags=OV, workspace=ws)
    torch.cuda.synchronize()
    r = check(q, k, v, o, lse, True, "bf16")
    assert r.passed, str(r)


def test_scheduler_slots_wrap_with_overlap():
    """More overlapped launches than scheduler slots (1024): every launch
    still claims every item."""
    q, k, v = _dev(*inputs.make_qkv(2, 32, 512, 512, 128, "bf16", 86))
    ref_o, ref_l = fa.fa_fwd(q, k, v, causal=True)
    o, lse = torch.empty_like(ref_o), torch.empty_like(ref_l)
    for _ in range(1100):
        fa.fa_fwd_ex(q, k, v, causal=True, flags=OV, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
