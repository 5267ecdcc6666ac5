"""Small, named launches of one kernel family each, for profiler captures.

    python -m exl3_trellis_weight_gb300.profile_cases encode --K 2 --rows 1216 --cols 256
    python -m exl3_trellis_weight_gb300.profile_cases rotate --rows 4096 --cols 4096
    python -m exl3_trellis_weight_gb300.profile_cases alu-mix
    python -m exl3_trellis_weight_gb300.profile_cases regularize --rows 4096 --cols 4096
    python -m exl3_trellis_weight_gb300.profile_cases ldl --rows 4096
    python -m exl3_trellis_weight_gb300.profile_cases ldlq --rows 1024 --cols 4096 --K 2
    python -m exl3_trellis_weight_gb300.profile_cases rows --rows 65536 --cols 160 --K 2

encode  : exl3_encode_tiles on fp32 N(0,1) targets (already rotated), scale 1.
rows    : exl3_encode_rows on fp32 N(0,1) targets: --rows rows of --cols (= T)
          targets each, scale 1.
rotate  : exl3_rotate (forward) of a bf16 N(0, 0.02^2) matrix.
alu-mix : build and run microbench/alu_mix.cu (instruction issue rates per SM
          per clock of the kinds the encoder uses).
regularize : exl3_regularize of a bf16 N(0, 0.02^2) matrix with a synthetic
          Hessian diagonal (inputs.hessian_diag).
ldl     : exl3_block_ldl of inputs.spd_hessian(rows) (rho 0.95).
ldlq    : exl3_ldlq of fp32 N(0, 1) targets with the factor of
          inputs.spd_hessian(rows), scale 1.
Each launch case runs --reps launches and synchronises; it prints the time per
launch from CUDA events on the current stream (and the wall time).  --copies N
(rotate) cycles N distinct input/output pairs, so that with N x 96 MiB above the
L2 size each launch reads its input from DRAM.
"""
from __future__ import annotations

import argparse
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None) -> int:
    import torch
    import exl3_trellis_weight_gb300 as ex
    from exl3_trellis_weight_gb300 import build, inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["encode", "rows", "rotate", "alu-mix", "regularize", "ldl", "ldlq"])
    ap.add_argument("--K", type=int, default=2)
    ap.add_argument("--rows", type=int, default=1216)
    ap.add_argument("--cols", type=int, default=256)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--copies", type=int, default=1)
    a = ap.parse_args(argv)
    if a.case == "alu-mix":
        import subprocess
        src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "microbench", "alu_mix.cu")
        exe = os.path.join(build.BUILD, "alu_mix")
        os.makedirs(build.BUILD, exist_ok=True)
        subprocess.run([build.nvcc(), *build.ARCH, "-O3", src, "-o", exe], check=True)
        return subprocess.run([exe]).returncode
    build.build()
    dev = torch.device("cuda:0")
    if a.case == "encode":
        Y = inputs.iid_f32(a.rows, a.cols, 0).to(dev)
        n = (a.rows // 16) * (a.cols // 16)
        ws = torch.empty(ex.encode_workspace_bytes(n, a.K), dtype=torch.uint8, device=dev)
        codes = torch.empty(a.rows // 16, a.cols // 16, 16 * a.K, dtype=torch.int16, device=dev)
        fn = lambda: ex.encode_tiles(Y, a.K, 1.0, codes=codes, ws=ws)
    elif a.case == "rows":
        Y = inputs.iid_f32(a.rows, a.cols, 0).to(dev)
        ws = torch.empty(ex.encode_workspace_bytes(a.rows, a.K), dtype=torch.uint8, device=dev)
        codes = torch.empty(a.rows, a.cols * a.K // 16, dtype=torch.int16, device=dev)
        fn = lambda: ex.encode_rows(Y, a.K, 1.0, codes=codes, ws=ws)
    elif a.case == "regularize":
        W = inputs.linear_bf16(a.rows, a.cols, 0).to(dev)
        h = inputs.hessian_diag(a.rows, 0).to(dev)
        sv = inputs.signs(a.cols, 2).to(dev)
        out = torch.empty(a.rows, a.cols, dtype=torch.float32, device=dev)
        ws = torch.empty(ex.regularize_workspace_bytes(a.rows, a.cols), dtype=torch.uint8, device=dev)
        fn = lambda: ex.regularize(W, h, sv, W_out=out, ws=ws)
    elif a.case in ("ldl", "ldlq"):
        H = inputs.spd_hessian(a.rows, 0, rho=0.95).to(dev)
        M = torch.empty(a.rows, a.rows, dtype=torch.float32, device=dev)
        wl = torch.empty(ex.block_ldl_workspace_bytes(a.rows), dtype=torch.uint8, device=dev)
        ex.block_ldl(H, M=M, ws=wl)
        if a.case == "ldl":
            fn = lambda: ex.block_ldl(H, M=M, ws=wl)
        else:
            del wl
            R = inputs.iid_f32(a.rows, a.cols, 0).to(dev)
            wq = torch.empty(ex.ldlq_workspace_bytes(a.rows, a.cols, a.K), dtype=torch.uint8,
                             device=dev)
            codes = torch.empty(a.rows // 16, a.cols // 16, 16 * a.K, dtype=torch.int16, device=dev)
            fn = lambda: ex.ldlq(R, M, a.K, 1.0, want_q=False, codes=codes, ws=wq)
    else:
        Ws = [inputs.linear_bf16(a.rows, a.cols, c).to(dev) for c in range(a.copies)]
        su, sv = (t.to(dev) for t in inputs.sign_pair(a.rows, a.cols, 0))
        outs = [torch.empty(a.rows, a.cols, dtype=torch.float32, device=dev) for _ in range(a.copies)]
        turn = [0]

        def fn():
            c = turn[0] % a.copies
            turn[0] += 1
            return ex.rotate(Ws[c], su, sv, out=outs[c])
    if a.copies > 1:
        for _ in range(2 * a.copies):
            fn()                                    # warm-up: every copy resident once
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record()
    for _ in range(a.reps):
        fn()
    ev1.record()
    torch.cuda.synchronize()
    wall = 1e3 * (time.perf_counter() - t0) / a.reps
    print(f"{a.case}: {a.reps} launches, {ev0.elapsed_time(ev1) / a.reps:.4f} ms each (events), "
          f"{wall:.3f} ms each (wall)")
    return 0


if __name__ == "__main__":
    sys.exit(main())
