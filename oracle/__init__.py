"""CPU oracle of the fused MXFP4 x FP8 MoE forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or run anything here; the
product path (the CUDA library and its Python binding) never does.  The
oracle shares no code with the CUDA path.

Modules:
  formats  exact E2M1 / E4M3 / E8M0 / bf16 codecs (OCP MX v1.0 definitions)
  moe      the forward, step by step, in float64 / float32 numpy

Parity status of each function is recorded in its docstring; every function
is pinned by a ``-m "not gpu"`` test under tests/ (format tables against
independent libraries, routing against torch.topk, expansion invariants,
quantiser bounds, and the whole forward against a brute-force dense
per-expert formulation plus hand-computed golden cases).
"""
from . import formats, moe  # noqa: F401
