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
