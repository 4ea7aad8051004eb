"""GB300-native low-precision packed-varlen attention forward (FP8 E4M3 and NVFP4).

The compute lives in a C-ABI CUDA library (``libfa_lp.so``, header ``include/fa_lp.h``);
``precision_attention_diffusion_gb300.fa_lp`` is a thin ctypes binding over it that only
marshals torch device pointers, strides and streams. Import it explicitly:
``from precision_attention_diffusion_gb300 import fa_lp``.
"""
