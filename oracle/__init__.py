"""CPU oracle for the GPT-2 training step (test infrastructure only).

Only tests, the package smoke check and the bench's CPU-baseline leg may
import this package.  The product path never does.
"""
