"""The C ABI library builds, loads without a GPU, and exports every function
that include/hisparse.h declares; the binding declares the same names."""
import os
import re

import __graft_entry__ as G

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "include", "hisparse.h")


def _declared():
    src = open(HDR).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    G.build()
    import hisparse_top_sparse_gb300 as hs
    L = hs.lib()
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), f"{n} declared in hisparse.h but not exported"
    assert sorted(hs.EXPORTS) == names


def test_argument_errors_return_without_a_gpu():
    G.build()
    import ctypes
    import hisparse_top_sparse_gb300 as hs
    L = hs.lib()
    # invalid sizes are rejected on the host before anything touches a device
    assert L.hs_resolve_topk(None, None, None, 0, None, -1, 4, 64, 64, None, None, None,
                             None) == hs.HS_ERR_INVALID_ARG
    assert b"bad sizes" in L.hs_last_error_string()
    assert L.hs_sparse_attn_decode(None, None, 0, None, 1, 0, 1, ctypes.c_float(1.0), None,
                                   None, None, None) == hs.HS_ERR_INVALID_ARG
    assert L.hs_buffer_create(None, None) == hs.HS_ERR_INVALID_ARG
    fits = ctypes.c_int32(7)
    assert L.hs_step_overlap_fits(0, ctypes.byref(fits)) == hs.HS_ERR_INVALID_ARG
    assert L.hs_step_overlap_fits(16385, ctypes.byref(fits)) == hs.HS_ERR_INVALID_ARG
    assert L.hs_step_overlap_fits(64, None) == hs.HS_ERR_INVALID_ARG
    assert L.hs_swap_in(None, None, None, None, None, 0, 0, None, None, None,
                        None) == hs.HS_ERR_INVALID_ARG
    # mixed batch: negative cache sizes, a negative request count with flags
    assert L.hs_sparse_attn_decode_mixed(None, None, -1, None, 0, None, None, 0, None, 1, 1, 1,
                                         ctypes.c_float(1.0), None, None, None,
                                         None) == hs.HS_ERR_INVALID_ARG
    flags = ctypes.c_int32(1)
    assert L.hs_sparse_attn_decode_mixed(None, None, 0, None, 0, None, ctypes.byref(flags), -1,
                                         None, 1, 1, 1, ctypes.c_float(1.0), None, None, None,
                                         None) == hs.HS_ERR_INVALID_ARG
    assert L.hs_reclaim_resident(None, -1, 4, None, 1, None, None, None,
                                 None) == hs.HS_ERR_INVALID_ARG
    assert L.hs_reclaim_resident(None, 2, 4, None, 1, None, None, None,
                                 None) == hs.HS_ERR_INVALID_ARG
    assert b"NULL" in L.hs_last_error_string()
    # row backups: bad token strides are refused before any device work
    assert L.hs_backup_rows(1, None, None, None, None, 4, 6, 10, 10, None,
                            None) == hs.HS_ERR_INVALID_ARG
    assert b"token_stride" in L.hs_last_error_string()
    assert L.hs_backup_indexer(1, None, None, None, None, None, 4, 0, 4, 16, 10, 10, None,
                               None) == hs.HS_ERR_INVALID_ARG
    # the bounded-wait check: a NULL status word or a limit out of range
    assert L.hs_wait_probe(None, 1000, None) == hs.HS_ERR_INVALID_ARG
    assert L.hs_wait_probe(ctypes.c_void_p(16), 0, None) == hs.HS_ERR_INVALID_ARG
    assert L.hs_wait_probe(ctypes.c_void_p(16), (1 << 31) + 1, None) == hs.HS_ERR_INVALID_ARG
    assert b"max_cycles" in L.hs_last_error_string()
