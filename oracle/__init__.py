"""FP64 CPU oracle for the shared-prefix one-pass decision path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it.  See oracle.py and blink_oracle.c.
"""
