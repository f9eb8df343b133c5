"""GB300-native weight-quantized GEMM (W4A16 INT4, W4A8 MXFP4, W4A4 NVFP4) and its grouped
MoE variant, behind the C ABI in include/hm.h.

``moe_hm_gemm_gb300.hm`` is the Python binding of ``libhm.so`` (argument marshalling only);
``moe_hm_gemm_gb300.synth`` holds the seeded synthetic input generators.
"""
__all__ = ["hm", "synth"]
