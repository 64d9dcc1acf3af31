"""The C-ABI library on the CPU: it loads, exports every entry point that
include/mp.h declares, and rejects bad arguments on the host before any
launch (no GPU needed; nothing here reaches a kernel)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from unpermute_routing_indices_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mp.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("mp_build_map", "mp_permute", "mp_unpermute", "mp_permute_bwd",
              "mp_unpermute_bwd", "mp_sort_chunks_pad", "mp_unpad_restore",
              "mp_sort_chunks_pad_bwd", "mp_unpad_restore_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_status_strings(lib):
    assert lib.mp_status_string(0) == b"ok"
    for code in (-1, -2, -3, -4):
        assert lib.mp_status_string(code) not in (b"ok", b"unknown status")


def test_workspace_size(lib):
    assert lib.mp_build_map_workspace_size(16384, 8, 128) % 256 == 0
    assert lib.mp_build_map_workspace_size(16384, 8, 128) >= 129 * 64 * 4
    assert lib.mp_build_map_workspace_size(0, 8, 128) == 256
    assert lib.mp_build_map_workspace_size(-1, 8, 128) == 0
    assert lib.mp_build_map_workspace_size(4, 8, 5000) == 0


FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: every call below fails validation


@pytest.mark.parametrize("args,code", [
    ((FAKE, -1, 4, 8, FAKE, None, FAKE, FAKE, FAKE, 4096, None, None), -1),   # T < 0
    ((FAKE, 4, 0, 8, FAKE, None, FAKE, FAKE, FAKE, 4096, None, None), -1),    # K < 1
    ((FAKE, 4, 2, 0, FAKE, None, FAKE, FAKE, FAKE, 4096, None, None), -1),    # E < 1
    ((FAKE, 4, 2, 5000, FAKE, None, FAKE, FAKE, FAKE, 4096, None, None), -3),  # E too big
    ((FAKE, 2**31, 2, 8, FAKE, None, FAKE, FAKE, FAKE, 4096, None, None), -3),  # R > int32
    ((None, 4, 2, 8, FAKE, None, FAKE, FAKE, FAKE, 4096, None, None), -1),    # idx NULL
    ((FAKE, 4, 2, 8, FAKE, None, None, FAKE, FAKE, 4096, None, None), -1),    # counts NULL
    ((FAKE, 4, 2, 8, FAKE, None, FAKE, FAKE, None, 4096, None, None), -2),    # no workspace
    ((FAKE, 4, 2, 8, FAKE, None, FAKE, FAKE, FAKE, 16, None, None), -2),      # too small
])
def test_build_map_rejects(lib, args, code):
    assert lib.mp_build_map(*args) == code


def test_row_ops_reject(lib):
    assert lib.mp_permute(None, None, FAKE, 4, 2, 8, FAKE, None, None) == -1
    assert lib.mp_permute(FAKE, FAKE, FAKE, 4, 2, 8, FAKE, None, None) == -1   # probs w/o out
    assert lib.mp_permute(FAKE, None, FAKE, 4, 2, 0, FAKE, None, None) == -1   # H < 1
    assert lib.mp_permute(FAKE, None, FAKE, 0, 2, 8, FAKE, None, None) == 0    # empty: no-op
    assert lib.mp_unpermute(FAKE, None, None, 4, 2, 8, FAKE, None) == -1
    assert lib.mp_permute_bwd(FAKE, FAKE, FAKE, 4, 2, 8, FAKE, None, None) == -1
    assert lib.mp_unpermute_bwd(FAKE, None, FAKE, FAKE, 4, 2, 8, FAKE, FAKE, None) == -1
    assert lib.mp_unpermute_bwd(FAKE, FAKE, FAKE, FAKE, 4, 2, 8, FAKE, None, None) == -1


def test_zero_rows_from_rejects(lib):
    assert lib.mp_zero_rows_from(None, 0, 64, None, None) == 0        # nothing to zero
    assert lib.mp_zero_rows_from(None, 10, 0, None, None) == 0
    assert lib.mp_zero_rows_from(None, 10, 64, FAKE, None) == -1
    assert lib.mp_zero_rows_from(FAKE, 10, 64, None, None) == -1
    assert lib.mp_zero_rows_from(FAKE, -1, 64, FAKE, None) == -1
    assert lib.mp_zero_rows_from(FAKE, 10, -2, FAKE, None) == -1
    assert lib.mp_zero_rows_from(FAKE, 1 << 40, 1 << 40, FAKE, None) == -1  # size overflow


def test_chunk_ops_reject(lib):
    ok = (FAKE, None, FAKE, FAKE, 128, 16, 128, 100, 200, 64, FAKE, None, FAKE, FAKE, None, None)
    bad_cg = list(ok); bad_cg[4] = 100                  # C % G != 0
    bad_al = list(ok); bad_al[6] = 0                    # align < 1
    big_c = list(ok); big_c[4] = 2048; big_c[5] = 16    # C > MP_MAX_CHUNKS
    no_gof = list(ok); no_gof[13] = None
    for args, code in ((bad_cg, -1), (bad_al, -1), (big_c, -3), (no_gof, -1)):
        assert lib.mp_sort_chunks_pad(*args) == code
    assert lib.mp_unpad_restore(FAKE, FAKE, FAKE, 10, 10, 8, FAKE, None, None, None) == -1
    assert lib.mp_unpad_restore(None, None, FAKE, 10, 10, 8, FAKE, None, None, None) == -1
    assert lib.mp_unpad_restore(FAKE, None, FAKE, 0, 10, 8, FAKE, None, None, None) == 0
    assert lib.mp_unpad_restore_bwd(FAKE, None, None, 10, 10, 8, FAKE, None, None, None) == -1
    assert lib.mp_sort_chunks_pad_bwd(FAKE, None, FAKE, -1, 10, 8, FAKE, None, None, None) == -1


@pytest.mark.parametrize("args,code", [
    ((FAKE, -1, 64, 8, 1, 1, FAKE, FAKE, None), -1),      # T < 0
    ((FAKE, 4, 64, 0, 1, 1, FAKE, FAKE, None), -1),       # K < 1
    ((FAKE, 4, 64, 33, 1, 1, FAKE, FAKE, None), -3),      # K > 32
    ((FAKE, 4, 2048, 8, 1, 1, FAKE, FAKE, None), -3),     # E > MP_MAX_EXPERTS
    ((FAKE, 4, 64, 8, 64, 1, FAKE, FAKE, None), -3),      # n_groups > 32
    ((FAKE, 4, 64, 8, 3, 1, FAKE, FAKE, None), -1),       # E % n_groups != 0
    ((FAKE, 4, 64, 8, 8, 9, FAKE, FAKE, None), -1),       # topk_groups > n_groups
    ((FAKE, 4, 64, 8, 16, 1, FAKE, FAKE, None), -1),      # kept experts < K
    ((FAKE, 4, 4, 8, 1, 1, FAKE, FAKE, None), -1),        # K > E
    ((FAKE, 0, 64, 8, 1, 1, None, None, None), 0),        # empty: no-op
    ((None, 4, 64, 8, 1, 1, FAKE, FAKE, None), -1),       # logits NULL
])
def test_router_rejects(lib, args, code):
    assert lib.mp_topk_softmax(*args) == code


def test_router_bwd_rejects(lib):
    assert lib.mp_topk_softmax_bwd(FAKE, FAKE, FAKE, 4, 64, 33, FAKE, None) == -3   # K > 32
    assert lib.mp_topk_softmax_bwd(FAKE, FAKE, FAKE, 4, 2048, 8, FAKE, None) == -3  # E too big
    assert lib.mp_topk_softmax_bwd(FAKE, FAKE, None, 4, 64, 8, FAKE, None) == -1    # idx NULL
    assert lib.mp_topk_softmax_bwd(None, None, None, 0, 64, 8, None, None) == 0     # empty


@pytest.mark.parametrize("args,code", [
    ((FAKE, None, FAKE, FAKE, 2**30, 4, 64, 64, 8, 0, FAKE, None), -1),   # T*K > int32
    ((FAKE, None, FAKE, FAKE, 4, 2, 64, 64, 6, 0, FAKE, None), -1),       # E % ep_size != 0
    ((FAKE, None, FAKE, FAKE, 4, 2, 64, 64, 0, 0, FAKE, None), -1),       # ep_size < 1
    ((FAKE, None, FAKE, FAKE, 4, 2, 64, 64, 8, 4, FAKE, None), -1),       # unknown flag
    ((FAKE, None, FAKE, FAKE, 4, 17, 64, 64, 8, 0, FAKE, None), -3),      # K > 16
    ((FAKE, None, FAKE, None, 4, 2, 64, 64, 8, 0, FAKE, None), -1),       # idx NULL
    ((None, None, None, None, 0, 2, 64, 64, 8, 3, None, None), 0),        # empty: no-op
])
def test_unpermute_ep_rejects(lib, args, code):
    assert lib.mp_unpermute_ep(*args) == code
