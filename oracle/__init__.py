"""CPU fp64 oracle for the routed-expert MLP (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Sources (cited by page title and section throughout):

* "Improving MoE training throughput with advanced fused kernels"
  (高度な融合カーネルによる MoE 学習スループットの向上), sections
  "Overcoming training bottlenecks in the MoE block",
  "Optimizing GLU activations with fused GEMM epilogues" (Figure 2),
  "Eliminating host-device synchronisation and CPU launch overhead",
  "Reducing exposed memory overhead by fusing MXFP8 and NVFP4 quantization",
  "From kernel-level gains to end-to-end pretraining speedups",
  "Next steps".
* "Accelerating dropless MoE training with JAX and NVIDIA Transformer
  Engine" (JAXとNVIDIA Transformer EngineによるDropless MoE学習の高速化),
  section "Claims and evidence" (grouped GEMM over ragged tensors).

The pages print no formulas; every definition here is the plain reading of
their prose, and each point they leave open is stated where it is used.

Parity status: every function is pinned by tests that do not re-run it
(brute force, closed forms, autograd of an independent forward, finite
differences, the MX format's own code table).  No function is unpinned.
"""
from .moe_oracle import *  # noqa: F401,F403
from .mx_oracle import *  # noqa: F401,F403
from .mx_mlp_oracle import *  # noqa: F401,F403
from .nvfp4_oracle import *  # noqa: F401,F403
