"""blink on GB300: the shared-prefix one-pass decision hot path as a C-ABI CUDA library.

Importing the package is cheap; the native library is loaded on first use of `lib()` or of
any entry point in `shared_prefix_question_gb300.blink`.
"""
__all__ = ["workloads", "blink"]
