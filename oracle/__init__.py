"""CPU oracle for the 2-bit sign-symmetric MoE expert layer with NVFP4 delta.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
fp64 (and, for tiny cases, exact-rational) restatement of what the GPU library
computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The CUDA library never calls it, never
links it and shares no code, table or helper with it; the only thing both
sides share is the seeded input generator in ``workloads.py``, which draws
random numbers and performs none of the method's arithmetic.

Sources: the vLLM-Moet README as captured on the pickgithub page ("Frontier
MoE on consumer Blackwell (SM120)"), sections "GLM-5.2 (753B) -- the headline
model" (modelopt NVFP4 format, load-time requantisation) and "How it fits --
2-bit experts at FP4 quality" (sign-symmetric 2-bit codebook, FP4 delta cache,
confidence gate).  The pages leave the exact 2-bit codebook open; this library
fixes q in {-3, -1, +1, +3} with an e4m3 scale per block of 16 along K.

Modules
  formats  exact e4m3 / e2m1 decoding and round-to-nearest-even
  nvfp4    fp32 -> NVFP4 quantiser (the input format of the experts)
  requant  NVFP4 -> 2-bit sign/magnitude planes, and the NVFP4 delta
  route    router top-k, renormalised softmax, bucketing permutation
  moe      the MoE forward (FC1 gate|up, SiLU*mul, FC2, weighted combine)
  gate     the confidence gate and the experts it promotes
  signbias the sign-bias probe (per-block L2-optimal fits to a 4-level codebook)

Every function here is pinned by a ``-m "not gpu"`` test in ``tests/`` to
something other than itself (brute force, closed forms, invariants, exact
rational arithmetic or a hand-worked example).  Agreement with the pages' own
outputs is unpinned: the pages print no tensors or layer outputs.
"""
from . import formats, nvfp4, requant, route, moe, gate, signbias  # noqa: F401
