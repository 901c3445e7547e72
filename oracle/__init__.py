"""Plain, slow, fp64 CPU oracle for the fused LoRA / QLoRA projection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA library in ``lora_qlora_linear_fwd_b300`` and the
library never imports it.
"""
from .lora_ref import *  # noqa: F401,F403
