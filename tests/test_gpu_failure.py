"""Failure detection on the GPU without faulting it.

A test-only build of the library (compiled with FA_TEST_SKIP_FIRST_Q) never
arms or loads the first Q tile of the prefill kernel, so the MMA warp's
bounded mbarrier wait runs out after about two seconds. The launch must then
report FA_ERR_TIMEOUT through the device error word, and the CUDA context must
stay usable for the normal library afterwards."""
import ctypes
import os
import tempfile

import numpy as np
import pytest
import torch

from gpu_util import assert_close, fa, run_prefill
from workloads import prefill_inputs

pytestmark = pytest.mark.gpu


def test_prefill_bounded_wait_reports_timeout(oracle_mod):
    from causal_gqa_flash_attn_gb300 import build, SIGNATURES
    m = fa()
    out_dir = os.path.join(tempfile.gettempdir(), "fa_test_skip_first_q")
    path = build.build(extra=["-DFA_TEST_SKIP_FIRST_Q"], out_dir=out_dir)
    L = ctypes.CDLL(path)
    for name in ("fa_prefill", "fa_get_device_error", "fa_kv_append", "fa_prefill_workspace_bytes"):
        res, args = SIGNATURES[name]
        getattr(L, name).restype = res
        getattr(L, name).argtypes = args

    n, hq, hkv, hd = 128, 2, 1, 64
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=5)
    kp = m.alloc_planes(1, m.KV_F32, hkv, n, hd)
    vp = m.alloc_planes(1, m.KV_F32, hkv, n, hd)
    pos0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd, vd = torch.from_numpy(k[None]).cuda(), torch.from_numpy(v[None]).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert L.fa_kv_append(kd.data_ptr(), vd.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                          pos0.data_ptr(), 1, n, hkv, hd, n, m.KV_F32, 0, 0, stream) == m.OK
    qd = torch.from_numpy(q).cuda()
    out = torch.zeros((n, hq, hd), device="cuda")
    ws = torch.empty(L.fa_prefill_workspace_bytes(n, hq, hkv, hd), dtype=torch.uint8, device="cuda")
    st = L.fa_prefill(qd.data_ptr(), kp.data_ptr(), vp.data_ptr(), out.data_ptr(), n, hq, hkv, hd,
                      0, 0, m.KV_F32, n, 0, 0, ws.data_ptr(), ws.numel(), None, stream)
    assert st == m.OK                                   # launched
    assert L.fa_get_device_error(stream) == m.ERR_TIMEOUT
    assert L.fa_get_device_error(stream) == m.OK       # read and cleared

    # the context is still healthy: the normal library computes correctly
    got = run_prefill(q, k, v, kv_fmt="f32", sink=0, win=0)
    assert_close(got, oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=0), "after timeout")
