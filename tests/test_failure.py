"""Failure path of the bounded waits, exercised on the GPU without a fault.

The self-test launch withholds every copy of a decode step, so each wait in
it runs into its 2 s bound; the kernel must record its code in the device
error word and end normally, after which the context must still compute
correct results."""

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import MODE_LSSAR, bf16_bits_to_f64, make_qkv
from oracle import attention_forward

pytestmark = pytest.mark.gpu

DECODE_WAIT_CODE = 41   # decode kernels: a wait for a stage that never landed


@pytest.fixture(scope="module")
def torch_mod():
    import torch
    from lssar_attn_fwd_gb300 import api, build
    build.build()
    api.load_library()
    return torch


def test_stalled_pipeline_reports_and_context_recovers(torch_mod):
    torch = torch_mod
    from lssar_attn_fwd_gb300 import api
    assert api.device_error_word() == 0          # clears any earlier code
    api.selftest_stall()
    assert api.device_error_word() == DECODE_WAIT_CODE
    assert api.device_error_word() == 0          # read clears it
    # the same process keeps working: a forward and a decode step vs the oracle
    qb, kb, vb = make_qkv(1, 2, 300, 64, seed=1)
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    out = api.lssar_attn_fwd(dev(qb), dev(kb), dev(vb), p=3, mode=MODE_LSSAR)
    dec = api.lssar_attn_decode(dev(qb[:, :, -1]), dev(kb), dev(vb), p=3, mode=MODE_LSSAR)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    ref = attention_forward(qf, kf, vf, MODE_LSSAR, 3)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= 2e-2
    assert np.abs(dec.float().cpu().numpy() - ref[:, :, -1]).max() <= 2e-2
