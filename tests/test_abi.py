"""The C-ABI library loads and exports every symbol include/*.h declares (no GPU, no compute calls)."""
import ctypes
import glob
import os
import re

from continuous_batching_paged_ragged_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(pkv_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(built):
    names = _declared()
    assert {"pkv_pool_init", "pkv_append", "pkv_attention", "pkv_sched_step"} <= names
    lib = ctypes.CDLL(pkv.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(built):
    assert _declared() <= set(pkv.SIGNATURES)


def test_host_side_argument_errors(built):
    """Errors detected on the host return a status before any launch (no GPU needed for these)."""
    bad = pkv.pkv_config(1, 4, 2, 64, 8, 64, 0)      # block_size 8 unsupported
    assert pkv.pkv_pool_bytes(bad) == 0
    ok = pkv.pkv_config(1, 4, 2, 64, 16, 64, 0)
    assert pkv.pkv_pool_bytes(ok) == 2 * 64 * 2 * 16 * 64 * 2 + 256
    odd = pkv.pkv_config(1, 6, 4, 64, 16, 64, 0)     # 6 % 4 != 0
    assert pkv.pkv_pool_bytes(odd) == 0
    h = ctypes.c_void_p()
    st = built.pkv_pool_init(ctypes.byref(ok), None, 0, ctypes.byref(h))
    assert st == pkv.PKV_ERR_INVALID_ARG and b"non-NULL" in built.pkv_last_error()
    assert built.pkv_append(None, 0, None, None, None, 1, None) == pkv.PKV_ERR_INVALID_ARG
    assert built.pkv_attention(None, 0, None, None, 1, None, None, 1, 1, None, None, 0, None) == pkv.PKV_ERR_INVALID_ARG


def test_8bit_pool_bytes_follow_the_header_layout(built):
    """Codes (one byte per value), then one scale byte per cached row, padded to 256, then the status area."""
    for layers, hkv, d, nb in [(1, 2, 64, 64), (3, 4, 128, 10), (2, 1, 256, 7)]:
        cfg = pkv.pkv_config(layers, 2 * hkv, hkv, d, 16, nb, 0, pkv.PKV_KV_E4M3)
        codes = 2 * layers * nb * hkv * 16 * d
        scales = 2 * layers * nb * hkv * 16
        assert pkv.pkv_pool_bytes(cfg) == (codes + scales + 255) // 256 * 256 + 256
        f16 = pkv.pkv_config(layers, 2 * hkv, hkv, d, 16, nb, 0, pkv.PKV_KV_F16)
        assert pkv.pkv_pool_bytes(f16) == 2 * codes + 256
    assert pkv.pkv_pool_bytes(pkv.pkv_config(1, 4, 2, 64, 16, 64, 0, 2)) == 0   # no such cache format
    assert built.pkv_pool_scales_ptr(None, 0) is None
