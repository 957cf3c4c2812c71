"""lbv_verify_fused_noalloc: the fused head with its argmax scratch in the
library module's own device memory.  Two calls in a row must give, bit for
bit, what lbv_verify_fused gives with a caller workspace, and the calls must
not change the device's free memory.  (Runs alone or after the other tests:
the scratch is zero at load and every call leaves it zero.)"""
import ctypes

import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import synth


def test_arguments_checked_before_any_device_work():
    L = lbv.lib()
    assert L.lbv_verify_fused_noalloc(None, None, 1, 1, None, lbv.FUSED_ARGMAX, None, None, 1,
                                      None, None, None) == lbv.ERR_INVALID_ARG
    assert "plan is NULL" in lbv.last_error()
    h = ctypes.c_void_p(1)      # never dereferenced: M is checked first
    assert L.lbv_verify_fused_noalloc(h, None, 9, 1, None, lbv.FUSED_ARGMAX, None, None, 1,
                                      None, None, None) == lbv.ERR_INVALID_ARG
    assert "8 rows" in lbv.last_error()


@pytest.mark.gpu
def test_noalloc_equals_workspace_call_two_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    K, N = 1280, 2000
    mat = synth.Matrix("w", synth.AFFINE2, K, N, 128, "f16", sigma_scale=0.01)
    parts, xb = synth.gen_matrix(mat, 31, rows=8)
    plan = lbv.Plan(lbv.FMT_AFFINE2, K, N, 128, lbv.F16)
    Wp = torch.from_numpy(lbv.pack(lbv.FMT_AFFINE2, parts, K, N, 128)).cuda()
    X1 = torch.from_numpy(xb.view(np.int16)).cuda()
    X2 = torch.from_numpy(synth.x_bits(np.random.default_rng(32), 8, K, "f16").view(np.int16)).cuda()
    ws = torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")
    ops = lbv.FUSED_ROTATE | lbv.FUSED_ARGMAX

    def outs():
        return (torch.full((8, N), -1.0, dtype=torch.float32, device="cuda"),
                torch.full((8,), -7, dtype=torch.int32, device="cuda"),
                torch.full((8,), -1.0, dtype=torch.float32, device="cuda"))

    for M, X in ((8, X1), (3, X2), (1, X1)):
        Ya, ia, va = outs()
        lbv.verify_fused(plan, X, M, Wp, ops, Y=Ya, idx=ia, val=va, workspace=ws)
        # two no-alloc calls in a row, one with logits and one without
        Yb, ib, vb = outs()
        _, ic, vc = outs()
        lbv.verify_fused_noalloc(plan, X, M, Wp, ops, Y=Yb, idx=ib, val=vb)
        lbv.verify_fused_noalloc(plan, X, M, Wp, ops, idx=ic, val=vc)
        torch.cuda.synchronize()
        plan.device_status()
        assert np.array_equal(Ya.cpu().numpy(), Yb.cpu().numpy())
        for i, v in ((ib, vb), (ic, vc)):
            assert np.array_equal(i.cpu().numpy(), ia.cpu().numpy())
            assert np.array_equal(v.cpu().numpy().view(np.uint32), va.cpu().numpy().view(np.uint32))
        assert np.all(ia.cpu().numpy()[M:] == -7)
    # without the argmax the call needs no scratch at all
    Yd, _, _ = outs()
    Ye, _, _ = outs()
    lbv.verify_fused(plan, X1, 8, Wp, lbv.FUSED_ROTATE, Y=Yd)
    lbv.verify_fused_noalloc(plan, X1, 8, Wp, lbv.FUSED_ROTATE, Y=Ye)
    torch.cuda.synchronize()
    assert np.array_equal(Yd.cpu().numpy(), Ye.cpu().numpy())
    # many calls leave the device's free memory as it was
    _, i0, v0 = outs()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(50):
        lbv.verify_fused_noalloc(plan, X1, 8, Wp, ops, idx=i0, val=v0)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
