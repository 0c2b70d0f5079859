"""VC-Attention for GB300 (sm_103a): V-Smooth preprocessing and the fused
low-bit attention forward, as hand-written CUDA behind a C ABI
(``include/vca.h``), with a thin Python binding (``vca``)."""
from . import vca  # noqa: F401
from .vca import (VCAttention, attention_bf16_ref, attention_fp8, attention_nvfp4,  # noqa: F401
                  get_status, state_bytes, state_layout, vsmooth_prepare)
