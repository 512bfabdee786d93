"""CPU oracle for the mixed-precision CA-SGD outer iteration (NumPy, FP64 / FP32).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or executes
this package: only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline /
reference arm of `bench.py` use it.  It shares no code with the CUDA path; the only
module both sides import is `synth_inputs` (seeded data, no method arithmetic).

Source: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
GPUs (abstract).  The abstract states the method in prose; the per-step formulas are
re-derived from plain minibatch SGD in `casgd.outer_step`'s docstring.

Every function here is pinned by a `-m "not gpu"` test (tests/test_oracle_*.py) to
something other than itself: published generator outputs, exact rational arithmetic,
closed forms, finite differences, the CA-SGD == s-step SGD identity, and NumPy /
PyTorch library routines.  The absolute final-loss values of the five workloads are
not printed anywhere on the pages: parity unpinned for those numbers.
"""
from .casgd import (  # noqa: F401
    LOGISTIC, LSQ, POISSON,
    splitmix64, sample_indices, bf16_round,
    perm_width, feistel, epoch_keys, permuted_indices, draw_indices,
    loss_value, loss_grad, full_loss,
    gram_block, gram_packed, packed_block_offset,
    outer_step, train, plain_sgd,
)
