"""CPU oracle for block-scaled FP8 (E4M3) video attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the test-suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  The CUDA
library shares no code with it: no kernels, headers, tables or helpers.

The oracle is plain, slow and written to be checked by eye against the pages
it follows.  All floating-point work is fp64 unless a step is defined at a
lower precision (the fp32 scale arithmetic of the prep, the E4M3 code itself,
the bf16 block means and outputs); those steps round exactly as stated.

Modules
  e4m3          bit-level OCP E4M3FN codec (round to nearest even, satfinite)
  bf16          exact rounding of real values to bfloat16
  prep          stage 1: Q/K block quantisation, V-Smooth gather/mean/residual quant
  attention     stage 2: emulated FP8 attention (exp2+cvt or ExpCast P-cast),
                exact fp64 attention, and the P-only emulation of the P-cast study
  closed_forms  P-underflow closed form, dp(S) sawtooth, reverse-order bound,
                error decomposition
  smooth        sequence-mean smoothing of K and V, V mean-bias correction
  cluster       online V clustering that produces the V-Smooth permutation
  nvfp4         4-bit PV product: E2M1 elements with a UE4M3 scale per 16 elements

Every function names the page and section it restates.  Where the pages leave
a step open the docstring states the reading taken.  Parity status: every
function here is pinned by a ``-m "not gpu"`` test against something other
than itself (see tests/test_oracle_*.py); none is "parity unpinned".  The
absolute MSE level of the P-cast study is pinned only loosely (within 35 %):
the pages print it without the V distribution behind it.
"""
