"""Plain CPU oracle for the routed-expert MoE decode layer (FP8 and NVFP4).

TEST INFRASTRUCTURE ONLY. This package is a slow, obviously-correct restatement
of what the pages define, in numpy with float64 sums. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it. The CUDA library under ``fp4_moe_expert_gb300`` never imports, links or
calls anything here, and nothing here imports the CUDA library: the two share
no code, tables or constants. Inputs reach both sides only through the seeded
generators in ``synth``.

Sources (cited by page title and section in every function):

* "vllm.models.glm5next.nvidia.specialized_decode.mega_moe" — ``MegaExperts``
  and ``_MegaKernel`` (routing ``top_k_pick``, ``_ordered``, the x-quant
  epilogue head, the GEMM1/GEMM2 epilogues, ``hidden_block``).
* "vllm.models.glm5next.nvidia.specialized_decode.shared_expert" —
  ``SharedExpert``, ``_GateUpKernel``, ``_DownKernel``, ``_group_scale``,
  ``block_scales``.
* "nvfp4-megamoe-kernel README.md" — "Data Formats", "Bugs Found & Fixed"
  sections 1, 2, 6 and 7 (slot pipeline, E2M1 staging, routing weights once).
* "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.comm" —
  ``EpCombine`` (the routing-weighted sum, FP32 in a fixed order, one BF16
  rounding): the local finalize; ``EpDispatch`` (MXFP8 quantiser) and the
  combine's rank-order reduction with RMSNorm, in their single-GPU forms.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
something other than itself (closed forms, exhaustive code tables, library
casts, brute force on tiny inputs, algebraic identities, invariants). No
function is "parity unpinned".
"""

from . import codecs, routing, quant, moe_fp8, moe_nvfp4, finalize, ep_local  # noqa: F401
