"""The index-checked build compiles without a GPU: libwenc_bounds.so (-DWENC_BOUNDS_CHECK) links
and exports exactly the entry points include/wenc.h declares, like libwenc.so."""
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "wenc.h")).read()
    return sorted(set(re.findall(r"WENC_API\s+[\w\s\*]+?\b(wenc_\w+)\s*\(", src)))


def test_bounds_checked_library_builds_and_exports_the_boundary():
    from transformer_encoder_gb300.build import LIB_BOUNDS, build
    path = build(bounds_check=True)
    assert path == LIB_BOUNDS and os.path.exists(path)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    syms = sorted({line.split()[-1] for line in out.splitlines() if line.split()[-1].startswith("wenc_")})
    assert syms == _declared()


def test_bounds_checks_vanish_from_the_normal_build():
    # the check helper is a compile-time no-op without the flag, a recorded, skipped access with it
    src = open(os.path.join(ROOT, "transformer_encoder_gb300", "csrc", "ptx.cuh")).read()
    assert "#ifdef WENC_BOUNDS_CHECK" in src and "in_bounds" in src
    for f in ("gemm.cu", "attn.cu"):
        assert "in_bounds(" in open(os.path.join(ROOT, "transformer_encoder_gb300", "csrc", f)).read()
