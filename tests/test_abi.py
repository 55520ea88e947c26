"""The C ABI on the host: the library loads, exports every function the
header declares, and rejects bad arguments with a status code and a message
before touching the GPU (no call here reaches a kernel launch)."""

import ctypes as C

import pytest
import torch

from long_context_sparse_25_b300 import csa


def test_library_exports_every_header_function():
    names = csa.header_functions()
    assert set(names) >= {"csa_compress", "csa_index", "csa_topk", "csa_attend", "hca_attend",
                          "csa_forward", "csa_workspace_size", "csa_last_error"}
    for n in names:
        assert hasattr(csa.lib, n), n


def _p(**kw):
    base = dict(B=1, m=4, H=8, D_qk=64, D_v=32, H_I=2, d_I=16, k=8, window=4, scale=0.1)
    base.update(kw)
    return csa.Params(*base.values())


FAKE = 1 << 20  # a 16-byte aligned non-null address that is never dereferenced


def _rows(width, n_rows=100, dtype=csa.BF16, data=FAKE):
    return csa.Rows(dtype, data, None, None, n_rows, width, width)


def test_compress_rejects_bad_arguments():
    out = _rows(64)
    f = csa.lib.csa_compress
    assert f(FAKE, FAKE, csa.E4M3, FAKE, 1, 0, 400, 4, 64, 0, 10, C.byref(out), None) == -2
    assert f(FAKE, FAKE, csa.BF16, FAKE, 0, 0, 400, 4, 64, 0, 10, C.byref(out), None) == -1
    assert f(None, FAKE, csa.BF16, FAKE, 1, 0, 400, 4, 64, 0, 10, C.byref(out), None) == -1
    assert "x is NULL" in csa.lib.csa_last_error().decode()
    assert f(FAKE + 8, FAKE, csa.BF16, FAKE, 1, 0, 400, 4, 64, 0, 10, C.byref(out), None) == -3
    # entries pool tokens beyond the rows given
    assert f(FAKE, FAKE, csa.BF16, FAKE, 1, 0, 39, 4, 64, 0, 10, C.byref(out), None) == -1
    # output too short
    assert f(FAKE, FAKE, csa.BF16, FAKE, 1, 0, 4000, 4, 64, 0, 101, C.byref(out), None) == -1
    # empty range: nothing to do, no pointer needed, no launch
    assert f(None, None, csa.BF16, None, 1, 0, 0, 4, 64, 3, 3, C.byref(out), None) == 0


def test_index_and_topk_reject_bad_arguments():
    p = _p()
    keys = _rows(16)
    f = csa.lib.csa_index
    assert f(C.byref(p), FAKE, csa.BF16, None, FAKE, C.byref(keys), 0, 4, 101, FAKE, None) == -1
    assert f(C.byref(p), FAKE, csa.E4M3, None, FAKE, C.byref(keys), 0, 4, 100, FAKE, None) == -2
    bad = _p(H_I=0)
    assert f(C.byref(bad), FAKE, csa.BF16, None, FAKE, C.byref(keys), 0, 4, 100, FAKE, None) == -1
    assert f(C.byref(p), FAKE, csa.BF16, None, FAKE + 4, C.byref(keys), 0, 4, 100, FAKE, None) == -3
    assert csa.lib.csa_topk(C.byref(_p(k=0)), FAKE, 0, 4, 100, FAKE, None, 0, None) == -1
    assert csa.lib.csa_topk(None, FAKE, 0, 4, 100, FAKE, None, 0, None) == -1


def test_attend_checks_window_coverage_and_dtypes():
    p = _p()
    kv = _rows(64)
    raw = _rows(64, n_rows=10)
    f = csa.lib.csa_attend
    # window of positions 50..53 not inside raw rows 60..69
    assert f(C.byref(p), FAKE, csa.BF16, C.byref(kv), C.byref(raw), 60, FAKE, 53, 1, 13, FAKE,
             csa.BF16, None, 0, None) == -1
    assert "window" in csa.lib.csa_last_error().decode()
    assert f(C.byref(p), FAKE, csa.E4M3, C.byref(kv), C.byref(raw), 50, FAKE, 53, 1, 13, FAKE,
             csa.BF16, None, 0, None) == -2
    big = _p(D_v=600, D_qk=640)
    kv2 = _rows(640)
    assert f(C.byref(big), FAKE, csa.BF16, C.byref(kv2), C.byref(raw), 50, FAKE, 53, 1, 13, FAKE,
             csa.BF16, None, 0, None) == -2
    # e4m3 raw rows are not accepted
    rawq = _rows(64, n_rows=10, dtype=csa.E4M3)
    assert f(C.byref(p), FAKE, csa.BF16, C.byref(kv), C.byref(rawq), 50, FAKE, 53, 1, 13, FAKE,
             csa.BF16, None, 0, None) == -2


def test_workspace_query_and_forward_workspace_check():
    p = _p(B=2)
    n = csa.lib.csa_workspace_size(C.byref(p), csa.WS_FORWARD, 3, 50)
    assert n >= 2 * 3 * 50 * 4 + 2 * 3 * 8 * 4
    assert csa.lib.csa_workspace_size(None, csa.WS_FORWARD, 3, 50) == 0
    a = csa.ForwardArgs()
    a.Q = 3
    a.q_pos0 = 197
    a.raw_dtype = csa.BF16
    a.kv = _rows(64)
    a.keys = _rows(16)
    assert csa.lib.csa_forward(C.byref(p), C.byref(a), FAKE, 16, None) == -4


def test_topk_workspace_covers_the_long_row_scratch():
    """The top-k workspace: nothing for rows the one-CTA-per-row path takes
    (N <= 16384, or 256 rows and more, or k > 4096); for a few long rows, room
    for one 8-byte (key, index) candidate per score, the per-row threshold and
    the per-list counts (at most 256 slices x 16 lists per row), each region
    rounded up to 256 bytes."""
    for (B, Q, N, k) in [(32, 1, 262144, 1024), (1, 1, 262144, 1024), (4, 1, 20001, 1024),
                         (64, 1, 131072, 1024), (1, 5, 20000, 1024), (255, 1, 20000, 1024)]:
        p = _p(B=B, k=k)
        ws = csa.workspace_size(p, csa.WS_TOPK, Q, N)
        rows = B * Q
        r256 = lambda x: (x + 255) // 256 * 256
        lo = r256(rows * 4) + r256(rows * 16 * 4) + r256(rows * N * 8)
        hi = r256(rows * 4) + r256(rows * 256 * 16 * 4) + r256(rows * N * 8)
        assert lo <= ws <= hi, (B, Q, N, k, ws)
    for (B, Q, N, k) in [(2, 3, 16384, 1024), (256, 1, 20000, 1024), (1, 1, 262144, 8192),
                         (1, 65536, 16384, 1024)]:
        assert csa.workspace_size(_p(B=B, k=k), csa.WS_TOPK, Q, N) == 0, (B, Q, N, k)


def test_debug_stall_aid_validates_its_argument():
    """csa_debug_stall_next touches no GPU state: it only arms a one-shot."""
    from long_context_sparse_25_b300 import csa
    assert csa.lib.csa_debug_stall_next(99) == -1
    assert csa.lib.csa_debug_stall_next(-1) == -1
    assert csa.lib.csa_debug_stall_next(0) == 0


def test_group_proj_rejects_bad_arguments():
    f = csa.lib.csa_group_proj
    # o [T=10, H=128, D_v=512], w [G=8, d_g=256, 8192], y [10, 2048]
    assert f(FAKE, 10, 128, 512, FAKE, 3, 256, FAKE, csa.BF16, None) == -1  # H % G
    assert "multiple of G" in csa.lib.csa_last_error().decode()
    assert f(FAKE, 10, 128, 512, FAKE, 8, 200, FAKE, csa.BF16, None) == -2  # d_g % 256
    assert f(FAKE, 10, 8, 12, FAKE, 8, 256, FAKE, csa.BF16, None) == -2     # K = 12
    assert f(FAKE, 10, 128, 512, FAKE, 8, 256, FAKE, csa.E4M3, None) == -2  # y dtype
    assert f(None, 10, 128, 512, FAKE, 8, 256, FAKE, csa.BF16, None) == -1
    assert f(FAKE + 8, 10, 128, 512, FAKE, 8, 256, FAKE, csa.BF16, None) == -3
    assert f(FAKE, -1, 128, 512, FAKE, 8, 256, FAKE, csa.BF16, None) == -1
    # T = 0: nothing to do, no pointer needed, no launch
    assert f(None, 0, 128, 512, None, 8, 256, None, csa.BF16, None) == 0


def test_fp4_key_rows_are_accepted_only_as_indexer_keys():
    p = _p()
    fp4 = csa.Rows(csa.E2M1, FAKE, None, FAKE, 100, 16, 16)
    f = csa.lib.csa_index
    # q_idx must be e4m3 with FP4 keys
    assert f(C.byref(p), FAKE, csa.BF16, None, FAKE, C.byref(fp4), 0, 4, 100, FAKE, None) == -2
    # odd width, missing scale
    odd = csa.Rows(csa.E2M1, FAKE, None, FAKE, 100, 15, 15)
    p15 = _p(d_I=15)
    assert f(C.byref(p15), FAKE, csa.E4M3, FAKE, FAKE, C.byref(odd), 0, 4, 100, FAKE, None) == -1
    noscale = csa.Rows(csa.E2M1, FAKE, None, None, 100, 16, 16)
    assert f(C.byref(p), FAKE, csa.E4M3, FAKE, FAKE, C.byref(noscale), 0, 4, 100, FAKE, None) == -1
    assert "scale" in csa.lib.csa_last_error().decode()
    # not as attention rows
    kv = csa.Rows(csa.E2M1, FAKE, None, FAKE, 100, 64, 64)
    raw = _rows(64, n_rows=10)
    assert csa.lib.csa_attend(C.byref(p), FAKE, csa.BF16, C.byref(kv), C.byref(raw), 50, FAKE, 53,
                              1, 13, FAKE, csa.BF16, None, 0, None) == -2
