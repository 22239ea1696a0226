"""CPU oracle of the MoE FFN layer forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never calls it, and it shares no code with the product: no
kernels, helpers, tables or constants.  Only the seeded input generators in
``workload/`` (which hold none of the layer's arithmetic) serve both.

Plain, slow and single-threaded in spirit: numpy float64, one step per
function, in the order the layer is defined.  See ``moe.py`` for the bf16
layer, ``fp8.py`` for the e4m3 codec and block quantisation, and
``nvfp4.py`` for the E2M1 codec, NVFP4 two-level block quantisation and the
NVFP4 layer.

Sources (page title, section):
  * ASAP: A DiSaggregated and Asynchronous Inference System for MoE Prefill,
    section 2.1 (experts as sparse sub-networks, a fraction active per
    token), section 3.4.2 (the MoE kernel is a grouped matrix multiplication,
    hidden states left, the layer's expert weights right), section 5.1
    (DeepSeek: 256 experts + 1 shared expert, 8 experts active per token),
    table 2 (per-expert token counts in the dispatch metadata).
  * DWDP: Distributed Weight Data Parallelism for High-Performance LLM
    Inference on NVL72, section 4.2 (grouped GEMM that reads a list of
    separately allocated per-expert weight buffers, no merge copy).
  * Memory-Compute Disaggregation for Large-Model Inference: AFD Architecture
    Analysis and Performance Validation, section 3, "Data-Flow Closed Loop"
    step 3 (FFN side: gated routing + expert computation).
The pages do not fix the scoring rule, SwiGLU, the routed scale, tie-breaks,
the permutation order, the fp8 scale convention or how NVFP4 activations
are scaled; those readings are stated where they are used.

Parity status: every function here is pinned by the CPU tests in
``tests/test_oracle_*.py`` (closed forms, invariants, brute force, hand-worked
fixtures under ``tests/golden/`` and library routines).  The fp8 scale
convention (amax/448 in fp32) and the NVFP4 tensor scales (amax/2688 for
weights, static per-layer scales for activations) are the readings that
nothing on the pages pins: "parity unpinned" beyond self-consistency and the
published codecs (OCP e4m3, OCP MX E2M1).
"""
from . import fp8, moe, nvfp4

__all__ = ["moe", "fp8", "nvfp4"]
