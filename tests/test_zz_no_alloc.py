"""fa_fwd_decode_static: the decode pass for callers that cannot allocate
device memory (its split partials live in the library's static device
scratch instead of a cudaMalloc'd workspace).  Collected last on purpose, so
a run that stops at the first failure has already run every other test.

Checked through the C ABI against the existing decode entry point (fa_fwd):
both run the same kernels with the same split on the same inputs, so on two
calls in a row with different inputs (the second call reuses the scratch the
first one left behind) the outputs must be equal bit for bit; the static
path is also gated against the fp64 oracle directly.  A shape whose partials
exceed the static scratch is rejected up front."""
import ctypes

import pytest
import torch

from attention_forward_gb300 import fa, inputs

pytestmark = pytest.mark.gpu

O_TOL = {"bf16": 2e-2, "fp16": 4e-3}   # the gate's absolute caps on O
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _static_call(q, k, v):
    B, H, _, D = q.shape
    Skv = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device=q.device)
    st = fa.load().fa_fwd_decode_static(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
        B, H, Skv, D, ctypes.c_float(D ** -0.5), fa._DTYPE[q.dtype],
        torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse


@pytest.mark.parametrize("B,H,Skv,D,dt", [(32, 32, 8192, 128, "bf16"),
                                         (3, 5, 1000, 64, "fp16")])
def test_two_calls_in_a_row_match_fa_fwd(B, H, Skv, D, dt):
    assert fa.fa_workspace_bytes(B, H, 1, Skv, D) > 0  # the split path runs
    for seed in (31, 32):
        q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, 1, Skv, D, dt, seed, 2.0))
        o_s, l_s = _static_call(q, k, v)
        o_r, l_r = fa.fa_fwd(q, k, v)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        # the same kernels, split and inputs: identical bits (a partial left
        # over from the previous call in the shared scratch would show here)
        assert torch.equal(o_s, o_r) and torch.equal(l_s, l_r), seed
        assert (o_s.float() - o_r.float()).abs().max().item() <= O_TOL[dt]
        assert (l_s - l_r).abs().max().item() <= LSE_TOL


def test_static_path_passes_the_oracle_gate():
    """The static entry point's own output against the fp64 oracle (all rows,
    the parity gate), after a call on other inputs has filled the scratch."""
    from parity import check
    B, H, Skv, D, dt = 4, 8, 3000, 128, "bf16"
    assert fa.fa_workspace_bytes(B, H, 1, Skv, D) > 0
    q0, k0, v0 = (t.cuda() for t in inputs.make_qkv(B, H, 1, Skv, D, dt, 40, 3.0))
    _static_call(q0, k0, v0)
    q, k, v = inputs.make_qkv(B, H, 1, Skv, D, dt, 41)
    o, lse = _static_call(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    r = check(q, k, v, o, lse, False, dt)
    assert r.passed, str(r)


def test_too_large_for_the_static_scratch_is_rejected():
    B, H, Skv, D = 64, 64, 1 << 20, 128
    need = fa.fa_workspace_bytes(B, H, 1, Skv, D)
    assert need > (8 << 20)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    st = fa.load().fa_fwd_decode_static(p, p, p, p, p, B, H, Skv, D,
                                        ctypes.c_float(0.088), fa.FA_BF16, None)
    assert st == fa.FA_ERR_WORKSPACE
