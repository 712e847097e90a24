"""lssar_attn_fwd_noalloc: the entry point that allocates no device memory.

Some callers cannot let a library allocate device memory during a call --
inference-runtime plugins whose enqueue step must not allocate, hosts that
reserve their whole memory budget at start-up, latency-critical loops where an
allocation could block on the driver.  For them the library keeps its scratch
in one fixed device array (LSSAR_NOALLOC_SCRATCH_BYTES per GPU).  These tests
call that entry point through the C ABI and check it against lssar_attn_fwd.

This file is named so that pytest collects it last.
"""

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import MODE_LSSA, MODE_LSSAR, MODE_SOFTMAX, make_qkv

SCRATCH_STATUS = -9


@pytest.fixture(scope="module")
def lib():
    from lssar_attn_fwd_gb300 import api, build
    build.build()
    return api.load_library()


def test_rejects_problems_beyond_the_fixed_scratch(lib):
    # B*H*L*d = 64M elements needs 256 MiB of scratch: rejected before any CUDA
    # call (the fake, far-apart pointers are never dereferenced).
    from lssar_attn_fwd_gb300.api import call_raw, status_string
    q, k, v, out = 1 << 36, 2 << 36, 3 << 36, 4 << 36
    st = call_raw("lssar_attn_fwd_noalloc", q, k, v, out, 1, 64, 8192, 128, 3, MODE_LSSAR, 0)
    assert st == SCRATCH_STATUS
    assert "scratch" in status_string(st)
    # ordinary argument errors keep their own codes
    assert call_raw("lssar_attn_fwd_noalloc", 0, k, v, out, 1, 1, 16, 64, 3, MODE_LSSAR, 0) == -1
    assert call_raw("lssar_attn_fwd_noalloc", q, k, v, out, 1, 1, 16, 96, 3, MODE_LSSAR, 0) == -3


@pytest.mark.gpu
@pytest.mark.parametrize("shape,mode,p", [
    ((1, 12, 1024, 64), MODE_LSSAR, 15),
    ((2, 4, 700, 128), MODE_LSSAR, 3),
    ((1, 2, 300, 64), MODE_LSSA, 1),
    ((2, 3, 257, 64), MODE_SOFTMAX, 1),
])
def test_matches_default_entry_point_on_two_calls(lib, shape, mode, p):
    # Both entry points run the same deterministic kernels on the same inputs
    # (only where the scratch lives differs), so the outputs must agree bit
    # for bit; a stale or shifted scratch would show up as any difference.
    import torch
    from lssar_attn_fwd_gb300 import api
    qb, kb, vb = make_qkv(*shape, seed=11)
    q, k, v = (torch.from_numpy(t.view(np.int16)).view(torch.bfloat16).cuda() for t in (qb, kb, vb))
    ref = api.lssar_attn_fwd(q, k, v, p=p, mode=mode)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):   # the second call reuses the array left by the first
        out = torch.full_like(q, float("nan"))
        st = api.call_raw("lssar_attn_fwd_noalloc", q.data_ptr(), k.data_ptr(), v.data_ptr(),
                          out.data_ptr(), *shape, p, mode, stream)
        assert st == 0, api.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert api.device_error_word() == 0
