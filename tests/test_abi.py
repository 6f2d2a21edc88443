"""The C-ABI library loads and exports every function include/fcp.h declares (no GPU needed)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "fcp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fcp_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("fcp_partition", "fcp_distribute", "fcp_block_attn_fwd", "fcp_block_attn_merge", "fcp_block_attn_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(fcp):
    handle = ctypes.CDLL(fcp.library_path())
    missing = [n for n in _declared() if not hasattr(handle, n)]
    assert not missing, missing
    # the binding binds exactly the declared set
    assert sorted(fcp.EXPORTED_SYMBOLS) == _declared()


def test_status_strings(fcp):
    L = fcp.lib()
    for s in range(7):
        assert L.fcp_status_string(s)
    assert L.fcp_last_error() is not None


def test_device_calls_validate_before_touching_the_gpu(fcp):
    """Argument errors come back as status codes, with no CUDA call made."""
    L = fcp.lib()
    p = fcp.Plan([300, 1024], 512, True)
    assert L.fcp_block_attn_fwd(p.handle, None, None, None, None, 4, 2, 64, None, None, None) == 1  # null d_plan
    assert L.fcp_plan_upload(p.handle, ctypes.c_void_p(256), 1 << 20, None) == 5  # not distributed
    p.distribute(2)
    d = ctypes.c_void_p(256)
    assert L.fcp_block_attn_fwd(p.handle, d, d, d, d, 4, 3, 64, d, d, None) == 1  # Hq % Hkv
    assert L.fcp_block_attn_fwd(p.handle, d, d, d, d, 4, 2, 96, d, d, None) == 3  # D unsupported
    assert L.fcp_block_attn_merge(p.handle, d, d, d, 4, 32, d, d, None) == 3
    assert L.fcp_plan_upload(p.handle, ctypes.c_void_p(257), 1 << 20, None) == 1  # misaligned
    assert L.fcp_plan_upload(p.handle, d, 16, None) == 1  # too small
    assert L.fcp_block_attn_bwd(p.handle, d, d, d, d, d, d, d, 4, 2, 64, d, d, d, d, 16, None) == 1  # small ws
    assert L.fcp_device_error(None, None, None) == 1
