"""CPU oracle for the fused W4A16 mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA path (``w4a16_moe_gb300``), and the CUDA path
never feeds it inputs or expected values.

It is a plain, slow, obviously correct restatement of what the layer computes,
in float64, written from the three pages the method is described on:

* flashinfer PR #4255, "feat(moe): sync SM12x W4A16 fused MoE family to b12x
  HEAD" (the subject: NVFP4 / MXFP4 weights, bf16 activations, route packing,
  FC1 with fused SiLU-SwiGLU or ReLU^2, FC2 with the top-k sum in its store);
* b12x PR #136, "fix(gemm): restore capture-safe K6 small-M dispatch"
  (caller-owned buffers, capture safety);
* b12x PR #137, "fix(moe): realign mixed Trellis with QSRT ABI" (ABI
  contract tests).

The pages print no equations and no worked numbers.  Where they are silent
the oracle takes the plainest reading; every such reading is named in the
function that takes it.

Modules
-------
formats   E2M1 / E4M3 / E8M0 decoders and round-to-nearest encoders, bf16_rn.
quant     NVFP4 (e4m3_k16 + fp32 global scale) and MXFP4 (e8m0_k32)
          quantisers and dequantisers, nibble packing.
routing   route validity, expert_map remap, power-of-two capacity, stable
          route packing.
moe       the fused MoE layer itself.
linear    the dense W4A16 linear layer (one weight matrix, no routing).

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` against something other than itself (torch casts,
bit-field definitions, brute force, closed forms, a dense-MLP special case,
exact integer arithmetic and invariances).  No function is "parity unpinned".
"""

from . import formats, quant, routing, moe, linear  # noqa: F401
