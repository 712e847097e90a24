"""The debug-check build (liblssar_attn_fwd_debug.so, -DLSSAR_DEBUG_CHECKS).

Its kernels check every tensor-copy coordinate, TMEM lane and column range,
work item and global-store index against the tensors they touch, and record
a code (101-105) in the library's device error word instead of making a bad
access; nothing traps.  It stands in for a memory checker: on ragged lengths
in every mode (forward, training forward and backward, decode step) the
word must stay 0, and the outputs must equal the default build's bit for bit
(the checks change no arithmetic).
"""

import ctypes

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import (
    MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW, make_dout, make_qkv)


def test_debug_build_is_a_separate_library():
    from lssar_attn_fwd_gb300 import api, build
    assert build.lib_path(debug=True) != build.lib_path()
    assert api.lib_path(debug=True).endswith("liblssar_attn_fwd_debug.so")
    assert "-DLSSAR_DEBUG_CHECKS" in build.DEBUG_FLAGS


@pytest.fixture(scope="module")
def libs():
    import torch
    from lssar_attn_fwd_gb300 import api, build
    build.build()
    build.build(debug=True)
    return torch, api.load_library(), api.load_debug_library()


def error_word(lib):
    w = ctypes.c_uint(0)
    assert lib.lssar_device_error_word(ctypes.byref(w)) == 0
    return w.value


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


MODES = [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_LSSA, 1), (MODE_SOFTMAX, 1), (MODE_SOFTMAX_RW, 15),
         (MODE_SIGMOID_RW, 3)]


@pytest.mark.gpu
@pytest.mark.parametrize("L", [1, 129, 257, 513])
@pytest.mark.parametrize("d", [64, 128])
def test_no_check_fires_on_ragged_lengths(libs, L, d):
    torch, rel, dbg = libs
    B, H = 2, 3
    qb, kb, vb = make_qkv(B, H, L, d, seed=L + d)
    db = make_dout(B, H, L, d, seed=L + d)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()   # noqa: E731
    q, k, v, dout = (dev(t) for t in (qb, kb, vb, db))
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert error_word(dbg) == 0
    for mode, p in MODES:
        outs = []
        for lib in (rel, dbg):
            out = torch.empty_like(q)
            stats = torch.empty((B, H, L, 4), dtype=torch.float32, device="cuda")
            grads = [torch.empty_like(q) for _ in range(3)]
            dec = torch.empty((B, H, d), dtype=torch.bfloat16, device="cuda")
            assert lib.lssar_attn_fwd(ptr(q), ptr(k), ptr(v), ptr(out), B, H, L, d, p, mode, s) == 0
            out2 = torch.empty_like(q)
            assert lib.lssar_attn_fwd_train(ptr(q), ptr(k), ptr(v), ptr(out2), ptr(stats),
                                            B, H, L, d, p, mode, s) == 0
            assert lib.lssar_attn_bwd(ptr(q), ptr(k), ptr(v), ptr(dout), ptr(stats), *(ptr(g) for g in grads),
                                      B, H, L, d, p, mode, s) == 0
            qd = q[:, :, -1].contiguous()
            assert lib.lssar_attn_decode(ptr(qd), ptr(k), ptr(v), ptr(dec), B, H, L, d, p, mode, s) == 0
            torch.cuda.synchronize()
            outs.append([out, out2, stats] + grads + [dec])
        assert error_word(dbg) == 0, (mode, p)
        assert error_word(rel) == 0, (mode, p)
        for a, b in zip(*outs):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b), (mode, p)
