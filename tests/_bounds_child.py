"""Runs the small parity cases on the bounds-checked build of the library.

Started by tests/test_gpu_bounds.py in a process of its own, with
DISCO_GB300_BOUNDS_CHECKED=1 so that the binding loads the build compiled
with -DDISCO_DEBUG_BOUNDS.  Every case must pass its oracle comparison with a
clean status word (disco_device_status raises DISCO_ERR_DEVICE_BOUNDS after a
failed range check).  Then, to show that the checks fire, psi is handed to
the contractions with its element counts understated: every index stays
inside the real arrays, so nothing is read out of bounds, but the checks see
indices past the stated extents, skip those accesses and must report
DISCO_ERR_DEVICE_BOUNDS.  Prints one line "bounds-checked: <n> cases clean,
<m> understated-extent runs flagged".
"""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def main() -> int:
    assert os.environ.get("DISCO_GB300_BOUNDS_CHECKED") == "1"
    import torch

    import sparse_spherical_convolution_gb300 as lib
    from tests import test_gpu_contract as tc
    from tests import test_gpu_fp16 as th
    from tests import test_gpu_fused as tf
    from tests import test_gpu_psi as tp

    assert lib.library_path().endswith("_bounds.so"), lib.library_path()
    assert lib.disco_build_flags() & lib.DISCO_BUILD_DEBUG_BOUNDS, "not the bounds-checked build"
    lib.disco_device_status(clear=True)

    n = n_flag = 0
    small_psi = [c for c in tp.CASES if c[0][0] * c[0][1] <= 64 * 128]
    runs = [(tc.test_fwd_bwd_full_compare, tc.SMALL), (tf.test_fused_full_compare, tf.SMALL),
            (th.test_fp16_contractions, th.CONTRACT), (th.test_fp16_fused_and_gradients, th.FUSED),
            (tp.test_psi_bit_exact, small_psi), (tp.test_runs_are_consistent_with_union_layout, small_psi)]
    for fn, cases in runs:
        for case in cases:
            fn(lib, case)
            assert lib.disco_device_status() == 0, (fn.__name__, case)
            n += 1

    # understated extents: the checks must flag (and skip) what lies past them
    import math
    fields = ("nruns", "nftab", "nhval", "nnz", "ngtab", "ngrp_ent")
    seen = set()
    for gi, go, kind, nrad, cut, B, C in (((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64, 1, 130),
                                          ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 1, 33),
                                          ((10, 24, 0), (10, 12, 0), 0, 1, 0.9, 2, 3)):
        psi = lib.Psi(gi, go, kind, nrad, cut)
        K = psi.c.K
        g = torch.Generator().manual_seed(5)
        x = torch.randn((B, C, gi[0], gi[1]), generator=g).to(torch.bfloat16).cuda()
        G = torch.randn((B, C, K, go[0], go[1]), generator=g).to(torch.bfloat16).cuda()
        X = torch.empty((B, C, K, go[0], go[1]), dtype=torch.bfloat16, device="cuda")
        gx = torch.empty((B, C, gi[0], gi[1]), dtype=torch.bfloat16, device="cuda")
        for field in fields:
            bad = lib.disco_psi.from_buffer_copy(psi.c)
            setattr(bad, field, getattr(psi.c, field) // 2)
            lib.disco_fwd(bad, x, X, B, C)
            lib.disco_bwd(bad, G, gx, B, C)
            try:
                lib.disco_device_status(clear=True)
            except lib.DiscoError as e:
                assert e.status == lib.DISCO_ERR_DEVICE_BOUNDS, e
                seen.add(field)
                n_flag += 1
            else:
                # every forward path walks the runs of each output row
                assert field != "nruns", (gi, go, "runs past an understated count went unflagged")
            assert lib.disco_device_status(clear=True) == 0
        # the true extents are clean again
        lib.disco_fwd(psi.c, x, X, B, C)
        lib.disco_bwd(psi.c, G, gx, B, C)
        assert lib.disco_device_status(clear=True) == 0
    # between them the three shapes take the tensor-core and CUDA-core paths of
    # both directions, which read every one of these arrays
    assert seen == set(fields), sorted(set(fields) - seen)
    print(f"bounds-checked: {n} cases clean, {n_flag} understated-extent runs flagged")
    return 0


if __name__ == "__main__":
    sys.exit(main())
