"""The C-ABI library: it builds, loads, exports every entry point that
include/fa.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from attention_forward_gb300 import _build, fa
    _build.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_ex", "fa_workspace_bytes", "fa_fwd_host",
              "fa_host_staging_bytes", "fa_get_device_status",
              "fa_set_watchdog_ns", "fa_status_string", "fa_version",
              "fa_prefill_uses_pairs", "fa_release_workspaces",
              "fa_fwd_decode_static", "fa_prefill_tail_items"):
        assert n in names, n


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in fa.h but not exported"


def test_binding_constants_match_the_header():
    """Every FA_FLAG_*, status and dtype constant of include/fa.h has the
    same value in the Python binding, and the binding names no flag the
    header lacks."""
    from attention_forward_gb300 import fa
    text = open(HEADER).read()
    flags = {n: int(v, 16) for n, v in re.findall(r"#define (FA_FLAG_\w+) (0x[0-9a-fA-F]+)u", text)}
    assert len(flags) >= 10
    for n, v in flags.items():
        assert getattr(fa, n) == v, n
    assert {n for n in dir(fa) if n.startswith("FA_FLAG_")} == set(flags)
    assert len(set(flags.values())) == len(flags)  # no two flags share a bit
    for n, v in re.findall(r"\b(FA_(?:OK|ERR_\w+|F16|BF16))\s*=\s*(\d+)", text):
        assert getattr(fa, n) == int(v), n


def test_status_strings_and_version(lib):
    from attention_forward_gb300 import fa
    for st in range(6):
        assert fa.fa_status_string(st)
    assert fa.fa_status_string(99) == "unknown status"
    assert fa.fa_version() == 10300


def test_pair_selection_without_a_gpu(lib):
    """The CTA-pair choice on the host (no device: SM count unknown, the
    default rule assumes 152 SMs): forced and refused by the flags, never for
    D=64, decode or a key split, by default only for long rows."""
    from attention_forward_gb300 import fa
    P, S = fa.FA_FLAG_PAIR, fa.FA_FLAG_SINGLE_CTA
    assert fa.fa_prefill_uses_pairs(1, 1, 300, 300, 128, True, P)
    assert not fa.fa_prefill_uses_pairs(4, 16, 4096, 4096, 128, False, S)
    assert not fa.fa_prefill_uses_pairs(1, 1, 300, 300, 64, True, P)
    assert not fa.fa_prefill_uses_pairs(1, 1, 1, 300, 128, False, P)
    assert not fa.fa_prefill_uses_pairs(1, 1, 300, 300, 128, False, P, num_splits=2)
    assert fa.fa_prefill_uses_pairs(4, 16, 4096, 4096, 128, False)
    assert fa.fa_prefill_uses_pairs(8, 16, 2048, 2048, 128, False)
    assert fa.fa_prefill_uses_pairs(16, 16, 1024, 1024, 128, False)
    assert not fa.fa_prefill_uses_pairs(32, 16, 512, 512, 128, False)
    assert not fa.fa_prefill_uses_pairs(16, 16, 1024, 512, 128, False)
    assert not fa.fa_prefill_uses_pairs(4, 16, 4096, 4096, 128, True)
    assert fa.fa_prefill_uses_pairs(2, 16, 8192, 8192, 128, True)
    assert fa.fa_prefill_uses_pairs(1, 16, 16384, 16384, 128, True)
    assert not fa.fa_prefill_uses_pairs(1, 1, 4096, 4096, 128, False)  # 8 items
    # the tail split needs the device's pair occupancy: none without a GPU
    assert fa.fa_prefill_tail_items(4, 16, 4096, 4096, 128, False,
                                    flags=fa.FA_FLAG_TAIL_SPLIT) == 0


def _call(lib, q=16, k=16, v=16, o=16, lse=16, B=1, H=1, Sq=8, Skv=8, D=64,
          scale=0.125, causal=0, dtype=1):
    return lib.fa_fwd(q, k, v, o, lse, B, H, Sq, Skv, D, scale, causal, dtype,
                      None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), 1), (dict(o=0), 1), (dict(lse=0), 1),
    (dict(k=24), 1), (dict(v=8), 1),                  # misaligned
    (dict(B=0), 1), (dict(H=-1), 1), (dict(Sq=0), 1), (dict(Skv=0), 1),
    (dict(B=256, H=256), 1), (dict(Sq=(1 << 24) + 1), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("inf")), 1),
    (dict(scale=float("nan")), 1),
    (dict(D=96), 2), (dict(D=256), 2), (dict(dtype=2), 2), (dict(dtype=-1), 2),
])
def test_argument_errors_precede_any_cuda_call(lib, kw, want):
    """Validation happens before the device is touched, so it answers the
    same on a machine without a GPU."""
    assert _call(lib, **kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), 1), (dict(lse=0), 1), (dict(k=24), 1), (dict(B=0), 1),
    (dict(Skv=0), 1), (dict(scale=0.0), 1), (dict(D=96), 2), (dict(dtype=2), 2),
])
def test_static_decode_argument_errors_precede_any_cuda_call(lib, kw, want):
    """fa_fwd_decode_static checks its arguments as fa_fwd does, before it
    looks at the device or its scratch."""
    a = dict(q=16, k=16, v=16, o=16, lse=16, B=1, H=1, Skv=8, D=64, scale=0.125,
             dtype=1)
    a.update(kw)
    assert lib.fa_fwd_decode_static(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                                    a["H"], a["Skv"], a["D"], ctypes.c_float(a["scale"]),
                                    a["dtype"], None) == want


def test_workspace_and_staging_sizes(lib):
    from attention_forward_gb300 import fa
    assert fa.fa_workspace_bytes(1, 1, 128, 128, 128) == 0   # one key tile: no split
    assert fa.fa_workspace_bytes(4, 64, 4096, 4096, 128) == 0  # items fill the GPU
    assert fa.fa_workspace_bytes(1, 8, 256, 16384, 128, 1) == 0  # no split asked
    n = fa.fa_workspace_bytes(1, 8, 256, 16384, 128, 4)  # 4 key ranges: O and LSE
    assert n >= 4 * 8 * 256 * (128 + 1) * 4 and n % 256 == 0
    assert fa.fa_workspace_bytes(1, 8, 256, 16384, 128) > 0   # the library splits
    assert fa.fa_workspace_bytes(1, 1, 1, 8192, 128, 1) == 0  # one split
    n = fa.fa_workspace_bytes(2, 3, 1, 1000, 128, 4)
    per = 2 * 3 * 4
    assert n >= per * 128 * 4 + per * 4 and n % 256 == 0
    assert fa.fa_host_staging_bytes(1, 2, 128, 256, 64) >= (
        2 * 128 * 64 * 2 * 2 + 2 * 2 * 256 * 64 * 2 + 2 * 128 * 4)


def test_binding_rejects_bad_tensors():
    from attention_forward_gb300 import fa
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q.float(), q)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q[:, :, :, :32], q)
    with pytest.raises(ValueError):
        fa.fa_fwd(q.transpose(2, 3), q, q)


def test_product_path_does_not_touch_the_oracle():
    """The library and its binding never load the oracle: no import of it in
    the package, and no oracle symbol in the shared object."""
    pkg = os.path.join(ROOT, "attention_forward_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "liboracle" not in src, f
    from attention_forward_gb300 import _build, fa
    _build.build()
    lib = fa.load()
    for name in ("oracle_attention_rows", "floor_attention_rows", "oracle_probs"):
        assert not hasattr(lib, name), name
