"""Run with MOE_LIBRARY=profile (tests/test_gpu_profile.py): the profile build
of the library, attached to a slot array, runs layout, notify, bf16 and int8
dispatch, combine and the fused launch; every output is compared with the
oracle bit for bit and every instrumented kernel must have filled its slots.
Prints "profile ok". Test infrastructure only."""

import ctypes
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from combine_moe_layout_02_gb300 import inputs, moe  # noqa: E402
from tests import gpu_path as gp  # noqa: E402

KERNELS, CTAS, PHASES = 8, 4096, 16  # MOE_PROF_KERNELS, MOE_PROF_CTAS, MOE_PROF_PHASES
LAYOUT, NOTIFY, DISPATCH, DISPATCH_INT8, FUSED = 0, 1, 2, 3, 5


def main():
    assert os.environ.get("MOE_LIBRARY") == "profile"
    L = moe.lib()
    assert moe.LIB_PATH.endswith("libmoe_profile.so")
    L.moe_profile_attach.restype = ctypes.c_int32
    L.moe_profile_attach.argtypes = [ctypes.c_void_p, ctypes.c_int64]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    slots = torch.zeros(KERNELS * CTAS * PHASES, dtype=torch.int64, device=dev)
    assert L.moe_profile_attach(slots.data_ptr(), 8) == moe.MOE_ERR_INVALID_ARG  # too small
    assert L.moe_profile_attach(slots.data_ptr(), slots.numel() * 8) == moe.MOE_OK

    w = inputs.workload("p32_e256_t128_h1024", T=40)
    gpu = gp.run_gpu(w)
    lay, nt = gp.oracle_tables(w)
    gp.assert_tables_equal(gpu, lay, nt)
    gp.compare_dispatch(w, 0, gpu, nt)
    gp.compare_combine(w, gpu, nt)
    q = gp.run_gpu(w, quant=1, y_mode="int8expert")
    gp.compare_dispatch(w, 1, q, nt)

    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, 0)
    fb = moe.Buffers(shape, dev)
    fb.dispatch_fused(torch.from_numpy(w.x_bits.view(np.int16)).to(dev), torch.from_numpy(w.topk_idx).to(dev),
                      torch.from_numpy(w.topk_weights).to(dev))
    torch.cuda.synchronize()
    assert int(fb.err[0].item()) == 0
    np.testing.assert_array_equal(fb.send_head.cpu().numpy(), nt["send_head"])

    a = slots.view(KERNELS, CTAS, PHASES).cpu().numpy()
    for k, phases in ((LAYOUT, range(1, 8)), (NOTIFY, range(1, 8)), (DISPATCH, range(1, 4)), (FUSED, range(1, 6))):
        row = a[k, 0]
        assert row[0] > 0, (k, "no start stamp")  # %globaltimer, ns
        stamps = row[list(phases)]
        assert (stamps > 0).all() and (np.diff(stamps) >= 0).all(), (k, stamps)
    assert a[DISPATCH_INT8, 0, 0] > 0 and a[DISPATCH_INT8, :, 5].sum() > 0  # tokens of consumer 0
    assert (a[DISPATCH_INT8, :, 1:5].sum(axis=0) > 0).all()
    assert L.moe_profile_attach(None, 0) == moe.MOE_OK  # detached
    print("profile ok")


if __name__ == "__main__":
    main()
