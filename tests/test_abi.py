"""Host-only checks of the C ABI: the library builds, loads, exports every
declared symbol, and rejects invalid arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

# Fake, far-apart, 16-byte aligned addresses: only ever passed together with
# at least one invalid argument, so nothing is dereferenced or launched.
Q, K, V, OUT = 1 << 32, 2 << 32, 3 << 32, 4 << 32


@pytest.fixture(scope="module")
def lib():
    from lssar_attn_fwd_gb300 import build
    from lssar_attn_fwd_gb300 import api
    build.build()
    return api.load_library()


def declared_functions():
    names = []
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(lssar_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    assert "lssar_attn_fwd" in names and "lssar_status_string" in names


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"


def test_abi_version(lib):
    assert lib.lssar_abi_version() >= 10000


def call(lib, name="lssar_attn_fwd", q=Q, k=K, v=V, out=OUT, B=1, H=1, L=16, d=64, p=3, mode=2):
    from lssar_attn_fwd_gb300.api import call_raw
    return call_raw(name, q, k, v, out, B, H, L, d, p, mode, 0)


@pytest.mark.parametrize("name", ["lssar_attn_fwd", "lssar_attn_fwd_simt"])
def test_invalid_arguments(lib, name):
    assert call(lib, name, q=0) == -1
    assert call(lib, name, out=0) == -1
    assert call(lib, name, mode=5) == -5
    assert call(lib, name, mode=-1) == -5
    assert call(lib, name, B=0) == -2
    assert call(lib, name, H=-1) == -2
    assert call(lib, name, L=0) == -2
    assert call(lib, name, L=(1 << 24) + 1) == -2
    assert call(lib, name, B=1 << 20, H=1 << 20, L=1 << 10, d=64) == -2
    assert call(lib, name, d=96) == -3
    assert call(lib, name, d=256) == -3
    assert call(lib, name, p=0) == -4
    assert call(lib, name, p=1025) == -4
    assert call(lib, name, mode=3, p=0) == -4     # re-weighting on the softmax normaliser
    assert call(lib, name, mode=4, p=0) == -4     # sigmoid + L1 + re-weighting
    assert call(lib, name, q=Q + 8) == -6
    assert call(lib, name, v=V + 2) == -6
    assert call(lib, name, out=Q + 1024) == -8   # out overlaps q
    assert call(lib, name, out=K - 1024) == -8   # out's range runs into k


def test_status_strings(lib):
    from lssar_attn_fwd_gb300.api import status_string
    assert status_string(0) == "ok"
    assert "64 or 128" in status_string(-3)
    assert status_string(-99) == "unknown status"


def test_binding_rejects_non_cuda_tensors():
    torch = pytest.importorskip("torch")
    from lssar_attn_fwd_gb300.api import lssar_attn_fwd
    x = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        lssar_attn_fwd(x, x, x)


def test_missing_library_fails_loudly(monkeypatch):
    from lssar_attn_fwd_gb300 import api
    monkeypatch.setattr(api, "_LIB", None)
    monkeypatch.setattr(api, "lib_path", lambda: "/nonexistent/liblssar_attn_fwd.so")
    with pytest.raises(RuntimeError, match="no fallback"):
        api.load_library()


def test_heads_p_invalid_arguments(lib):
    from lssar_attn_fwd_gb300.api import call_heads_p
    good = [3, 15]
    assert call_heads_p(Q, K, V, OUT, 1, 2, 16, 64, [], 2, 0) == -1          # no array
    assert call_heads_p(Q, K, V, OUT, 1, 2, 16, 64, good, 0, 0) == -4        # softmax: no p
    assert call_heads_p(Q, K, V, OUT, 1, 2, 16, 64, good, 1, 0) == -4        # LSSA: no p
    assert call_heads_p(Q, K, V, OUT, 1, 2, 16, 64, good, 9, 0) == -5
    assert call_heads_p(Q, K, V, OUT, 1, 2, 16, 64, [3, 0], 2, 0) == -4
    assert call_heads_p(Q, K, V, OUT, 1, 2, 16, 64, [3, 2000], 3, 0) == -4
    assert call_heads_p(Q, K, V, OUT, 1, 300, 16, 64, [3] * 300, 2, 0) == -4  # > 256 heads
    assert call_heads_p(Q, K, V, OUT, 1, 2, 16, 96, good, 4, 0) == -3
    assert call_heads_p(Q + 4, K, V, OUT, 1, 2, 16, 64, good, 2, 0) == -6


def test_decode_invalid_arguments(lib):
    from lssar_attn_fwd_gb300.api import call_raw
    f = "lssar_attn_decode"
    assert call_raw(f, 0, K, V, OUT, 1, 2, 16, 64, 3, 2, 0) == -1
    assert call_raw(f, Q, K, V, OUT, 1, 2, 16, 64, 3, 7, 0) == -5
    assert call_raw(f, Q, K, V, OUT, 1, 2, 0, 64, 3, 2, 0) == -2
    assert call_raw(f, Q, K, V, OUT, 1, 2, 16, 32, 3, 2, 0) == -3
    assert call_raw(f, Q, K, V, OUT, 1, 2, 16, 64, 0, 3, 0) == -4
    assert call_raw(f, Q, K + 2, V, OUT, 1, 2, 16, 64, 3, 2, 0) == -6
    assert call_raw(f, Q, K, V, K + 64, 1, 2, 16, 64, 3, 2, 0) == -8   # out inside the key cache


def test_decode_plan_invalid_arguments(lib):
    import ctypes
    out = [ctypes.c_int(0) for _ in range(4)]
    refs = [ctypes.byref(v) for v in out]
    assert lib.lssar_decode_plan(0, 2, 16, 64, *refs) == -2
    assert lib.lssar_decode_plan(1, 2, 0, 64, *refs) == -2
    assert lib.lssar_decode_plan(1, 2, (1 << 24) + 1, 64, *refs) == -2
    assert lib.lssar_decode_plan(1, 2, 16, 96, *refs) == -3


STATS, DQ, DK, DV, DOUT = 5 << 32, 6 << 32, 7 << 32, 8 << 32, 9 << 32


def test_train_invalid_arguments(lib):
    from lssar_attn_fwd_gb300.api import call_train
    assert call_train(Q, K, V, OUT, 0, 1, 2, 16, 64, 3, 2, 0) == -1           # no stats
    assert call_train(0, K, V, OUT, STATS, 1, 2, 16, 64, 3, 2, 0) == -1
    assert call_train(Q, K, V, OUT, STATS + 4, 1, 2, 16, 64, 3, 2, 0) == -6   # stats alignment
    assert call_train(Q, K, V, OUT, Q + 256, 1, 2, 16, 64, 3, 2, 0) == -8     # stats inside q
    assert call_train(Q, K, V, OUT, STATS, 1, 2, 16, 64, 0, 2, 0) == -4
    assert call_train(Q, K, V, OUT, STATS, 1, 2, 16, 80, 3, 2, 0) == -3
    assert call_train(Q, K, V, OUT, STATS, 1, 2, 16, 64, 3, 6, 0) == -5


BWD_NAMES = ["lssar_attn_bwd", "lssar_attn_bwd_simt"]


@pytest.mark.parametrize("name", BWD_NAMES)
def test_backward_invalid_arguments(lib, name):
    from lssar_attn_fwd_gb300.api import call_bwd
    good = [Q, K, V, DOUT, STATS, DQ, DK, DV]

    def c(idx=None, val=None, B=1, H=2, L=16, d=64, p=3, mode=2):
        ptrs = list(good)
        if idx is not None:
            ptrs[idx] = val
        return call_bwd(name, ptrs, B, H, L, d, p, mode, 0)

    for idx in range(8):
        assert c(idx, 0) == -1, idx                  # every pointer is required
    assert c(mode=5) == -5
    assert c(L=0) == -2
    assert c(d=32) == -3
    assert c(p=0) == -4
    assert c(3, DOUT + 2) == -6
    assert c(4, STATS + 8) == -6
    assert c(7, DV + 4) == -6
    assert c(5, Q + 64) == -8                         # dq over q
    assert c(6, DOUT) == -8                           # dk over dout
    assert c(7, STATS) == -8                          # dv over the stats
    assert c(6, DQ + 256) == -8                       # dk overlaps dq


def test_train_and_backward_heads_p_invalid_arguments(lib):
    from lssar_attn_fwd_gb300.api import call_bwd_heads_p, call_train_heads_p
    good = [3, 15]
    t = lambda *a: call_train_heads_p(*a, 0)   # noqa: E731
    assert t(Q, K, V, OUT, STATS, 1, 2, 16, 64, [], 2) == -1            # no array
    assert t(Q, K, V, OUT, 0, 1, 2, 16, 64, good, 2) == -1              # no stats
    assert t(Q, K, V, OUT, STATS, 1, 2, 16, 64, good, 0) == -4          # softmax: no p
    assert t(Q, K, V, OUT, STATS, 1, 2, 16, 64, [3, 0], 2) == -4
    assert t(Q, K, V, OUT, STATS, 1, 300, 16, 64, [3] * 300, 2) == -4   # > 256 heads
    assert t(Q, K, V, OUT, STATS + 4, 1, 2, 16, 64, good, 2) == -6
    assert t(Q, K, V, OUT, Q + 256, 1, 2, 16, 64, good, 2) == -8        # stats inside q
    assert t(Q, K, V, OUT, STATS, 1, 2, 16, 96, good, 2) == -3
    ptrs = [Q, K, V, DOUT, STATS, DQ, DK, DV]
    b = lambda ptrs, H=2, d=64, pp=good, mode=2: call_bwd_heads_p(ptrs, 1, H, 16, d, pp, mode, 0)   # noqa: E731
    assert b(ptrs, pp=[]) == -1
    assert b(ptrs, mode=1) == -4
    assert b(ptrs, pp=[3, 1025]) == -4
    assert b(ptrs, d=32) == -3
    assert b(ptrs[:4] + [0] + ptrs[5:]) == -1                          # no stats
    assert b(ptrs[:5] + [Q + 64] + ptrs[6:]) == -8                     # dq over q


@pytest.mark.parametrize("BH,n_qtiles,grid", [(12, 64, 152), (96, 8, 152), (64, 32, 152), (12, 128, 152),
                                              (8, 64, 152), (1, 1, 1), (3, 5, 7), (5, 63, 152), (200, 2, 152)])
def test_schedule_covers_every_item_once(lib, BH, n_qtiles, grid):
    n_pairs = (n_qtiles + 1) // 2
    n_items = BH * n_pairs
    grid = min(grid, n_items)
    first = (ctypes.c_int * (2 * grid))()
    tail = ctypes.c_int(0)
    assert lib.lssar_schedule_plan(BH, n_qtiles, grid, first, ctypes.byref(tail)) == 0
    fixed = [x for x in first if x >= 0]
    assert len(fixed) == len(set(fixed))
    # the fixed items are exactly [0, tail); the counter serves [tail, n_items)
    assert sorted(fixed) == list(range(tail.value))
    assert 0 < tail.value <= n_items
    # every CTA's first fixed item (if any) is in slot 0
    assert all(first[2 * c] >= 0 or first[2 * c + 1] < 0 for c in range(grid))


def test_schedule_pairs_long_with_short_items(lib):
    # 12 heads of 8192 rows (64 Q tiles, 32 pairs) on 152 CTAs: the long items
    # come with complements, and the largest planned load is near the mean
    BH, n_qtiles, grid = 12, 64, 152
    first = (ctypes.c_int * (2 * grid))()
    tail = ctypes.c_int(0)
    assert lib.lssar_schedule_plan(BH, n_qtiles, grid, first, ctypes.byref(tail)) == 0
    cost = lambda i: 4 * (31 - i // BH) + 3   # noqa: E731  K tiles of the pair's two Q tiles
    loads = [sum(cost(x) for x in (first[2 * c], first[2 * c + 1]) if x >= 0) for c in range(grid)]
    mean = sum(cost(i) for i in range(BH * 32)) / grid
    assert tail.value > grid and max(loads) <= 1.02 * mean


def test_schedule_rejects_bad_arguments(lib):
    first = (ctypes.c_int * 2)()
    tail = ctypes.c_int(0)
    assert lib.lssar_schedule_plan(0, 4, 1, first, ctypes.byref(tail)) == -2
    assert lib.lssar_schedule_plan(1, 4, 300, first, ctypes.byref(tail)) == -2
    assert lib.lssar_schedule_plan(1, 4, 1, None, ctypes.byref(tail)) == -1
