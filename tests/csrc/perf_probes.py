"""Drivers for the timing probes in probe.cu (not run by pytest).

    python tests/csrc/perf_probes.py ops     issue rate of single instructions per SM
    python tests/csrc/perf_probes.py stage   throughput of the decode stage arithmetic
    python tests/csrc/perf_probes.py mma     tcgen05.mma cycles per instruction
    python tests/csrc/perf_probes.py launch  launch latency of an empty kernel inside a CUDA graph
    python tests/csrc/perf_probes.py subnormal  mma.sync bf16 with subnormal A inputs

Needs a GPU and tests/csrc/libb4probe.so (built by __graft_entry__.build()).
"""

import ctypes
import os
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = ctypes.CDLL(os.path.join(HERE, "libb4probe.so"))


def ops():
    f = LIB.probe_op_tput
    f.argtypes = [ctypes.c_int] * 3 + [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    names = ["prmt", "lop3", "mul.hi.u32", "mul.rn.bf16x2", "shr.b32", "fma.rn.f32", "mul.rn.f16x2",
             "fma.rn.bf16x2", "mad.lo.u32", "add.u32"]
    iters = 4096
    out = torch.zeros(sms * 256, dtype=torch.int32, device="cuda")
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    for op, nm in enumerate(names):
        assert f(op, 64, sms, 3, out.data_ptr(), cyc.data_ptr()) == 0
        assert f(op, iters, sms, 3, out.data_ptr(), cyc.data_ptr()) == 0
        rate = 8 * 8 * iters / cyc.double().mean().item()
        print(f"{nm:14s} {rate:.2f} warp-instructions / clock / SM")


def stage():
    f = LIB.probe_decode_stage
    f.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    stages = 4096
    names = ["as the decode kernel", "one stage per step", "dequantisation only", "MMAs only"]
    for per_sm, smem in ((1, 200 * 1024), (2, 104 * 1024), (3, 70 * 1024), (4, 53 * 1024)):
        grid = sms * per_sm
        out = torch.zeros(grid * 256, device="cuda")
        cyc = torch.zeros(grid, dtype=torch.int64, device="cuda")
        for v in range(4):
            assert f(v, 256, grid, smem, out.data_ptr(), cyc.data_ptr()) == 0
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            assert f(v, stages, grid, smem, out.data_ptr(), cyc.data_ptr()) == 0
            e.record()
            torch.cuda.synchronize()
            ms = s.elapsed_time(e)
            gbs = grid * stages * 4608 / (ms * 1e-3) / 1e9
            print(f"CTAs/SM {per_sm}, {names[v]:22s}: {gbs:6.0f} GB/s of 4-bit weights, "
                  f"{cyc.double().mean().item() / stages:5.0f} cycles / stage / CTA")


def mma():
    f = LIB.probe_mma_tput
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    for name, v in (("N=160, A tmem, 1 acc", 1), ("N=160, A smem, 1 acc", 2 | 1), ("N=160, A smem, 2 acc", 2 | 1 | 16),
                    ("N=256, A smem, 1 acc", 2 | 8), ("N=256, A smem, 2 acc", 2 | 8 | 16),
                    ("N=16,  A smem, 2 acc", 2 | 16),
                    ("SW128 N=64,  A smem, 2 acc", 32 | 2 | 16 | 128), ("SW128 N=128, A smem, 2 acc", 32 | 2 | 16 | 64),
                    ("SW128 N=256, A smem, 2 acc", 32 | 2 | 16 | 8), ("SW128 N=128, A tmem, 1 acc", 32 | 64),
                    ("SW128 N=256, A tmem, 1 acc", 32 | 8),
                    ("SW128 M=64 N=128, A smem, 2 acc", 256 | 32 | 2 | 16 | 64),
                    ("SW128 M=64 N=256, A smem, 2 acc", 256 | 32 | 2 | 16 | 8),
                    ("hoisted descriptors, N=64", 512 | 128), ("hoisted descriptors, N=128", 512 | 64),
                    ("hoisted descriptors, N=256", 512 | 8),
                    ("kernel-like loop (per-MMA descriptors, runtime slot, commit per stage), N=128", 2048 | 64),
                    ("  the same + two barrier waits and a fence per stage", 2048 | 8192 | 64),
                    ("  the same with A in tensor memory, no waits", 2048 | 16384 | 64),
                    ("  the same with A in tensor memory + waits", 2048 | 8192 | 16384 | 64),
                    ("  A in tensor memory, test_wait first + fence", 2048 | 32768 | 16384 | 64),
                    ("  A in tensor memory, try_wait, no fence", 2048 | 65536 | 16384 | 64),
                    ("kernel-like, A in tensor memory, no waits, three warps storing to TMEM meanwhile",
                     2048 | 16384 | 64 | 131072),
                    ("kernel-like, A in shared memory, no waits, three warps storing to TMEM meanwhile",
                     2048 | 64 | 131072)):
        for per, pc in ((4, 4), (4, 0)):
            assert f(v, per, pc, out.data_ptr(), st.data_ptr()) == 0
            assert f(v, per, pc, out.data_ptr(), st.data_ptr()) == 0
            t1, t2 = out.tolist()
            n = 64 * per
            commit = "one commit per 4" if pc else "no commits"
            print(f"{name}, {commit:16s}: {t1 / n:6.1f} cycles / MMA issued, {t2 / n:6.1f} to completion")


def subnormal():
    """mma.sync bf16 with subnormal A: 16 products of A x B summed per output."""
    f = LIB.probe_mma_sync_const
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    out = torch.zeros(128, device="cuda")
    for a_bits, what in ((0x0040, "2^-127 (subnormal)"), (0x0001, "2^-133 (smallest subnormal)"),
                         (0x0080, "2^-126 (smallest normal)"), (0x3F80, "1.0")):
        for b_bits, bwhat in ((0x7180, "2^100"), (0x3F80, "1.0")):
            assert f(a_bits, b_bits, out.data_ptr()) == 0
            v = out[0].item()
            print(f"A = {what:28s} B = {bwhat:6s}: D = {v!r} (all equal: {bool((out == out[0]).all())})")


def launch():
    f = LIB.probe_launch
    f.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for name, grid, block, smem, coop in (("1 x 32, no smem", 1, 32, 0, 0),
                                          (f"{2 * sms} x 352, 70 KB", 2 * sms, 352, 70 * 1024, 0),
                                          (f"{2 * sms} x 352, 70 KB, cooperative", 2 * sms, 352, 70 * 1024, 1),
                                          (f"{sms} x 512, 172 KB", sms, 512, 172 * 1024, 0)):
        with torch.cuda.stream(s):
            assert f(grid, block, smem, coop, out.data_ptr(), s.cuda_stream) == 0
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            assert f(grid, block, smem, coop, out.data_ptr(), s.cuda_stream) == 0
        times = []
        for i in range(30):
            with torch.cuda.stream(s):
                flush.zero_()  # keeps the GPU busy while the host queues the replay
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                g.replay()
                b.record(s)
            s.synchronize()
            if i >= 5:
                times.append(a.elapsed_time(b) * 1e3)
        times.sort()
        print(f"{name:40s}: median {times[len(times) // 2]:.2f} us per graph replay (event to event)")


if __name__ == "__main__":
    {"ops": ops, "stage": stage, "mma": mma, "launch": launch, "subnormal": subnormal}[sys.argv[1]]()
