"""CPU oracle for the weight-quantized GEMM (test infrastructure only).

This package is a plain, slow, fp64 restatement of what the GPU library computes:
quantizers, dequantizers, the packed-weight layout and the GEMM itself. It exists so
that tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` can
check the CUDA path against something independent. Nothing in the product path may
import it, and it shares no code with the CUDA kernels or their Python binding.

Method source: "Humming: fast, flexible kernels for quantized inference" as described
on the vLLM/Humming explainer page (portfolio.ywsung.com, "vLLM Humming은 4비트를
어떻게 계산하나"), sections on scales, weight preprocessing, M-dependence and MoE; and
the news pages (news.cocoloop.cn, aihaber.org) for the format list. Number formats are
taken from their public definitions (OCP Microscaling v1.0 for E8M0/e2m1/e4m3, NVFP4's
two-level scaling, IEEE-754 round-to-nearest-even).

Parity status of each function is stated in its module docstring. Every function here
is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py``.
"""
