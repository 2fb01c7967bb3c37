"""CPU oracle for sequence-parallel exact attention (TEST INFRASTRUCTURE ONLY).

This package is a plain, slow, fp64 NumPy statement of what the GPU library
computes. It exists so tests can check the CUDA path against something whose
correctness can be read off the page by eye. Only `tests/`, the package's
smoke check and the benchmark's CPU-baseline leg may import it; the library
itself never does, and it shares no code with the CUDA path.

Modules
  attention  exact masked softmax attention and its gradient (the definition)
  layouts    contiguous / zigzag / stripe sequence permutations and the
             Ulysses sequence<->head all-to-all, as index maps
  merge      the associative log-sum-exp merge of (O, LSE) partials
  ring       a ring simulator: per-chunk partials in ring order + merge
  decode     a decode step: the newest tokens against a sharded KV cache,
             and the per-shard partials that a tree merge combines
  fp8        E4M3 codes (encode / decode / per-tensor quantization) and the
             attention of e4m3 q, k, v with per-tensor descales

Every function is pinned by `-m "not gpu"` tests against something other than
itself (brute force, a library routine, finite differences, closed forms and
the worked examples printed on the pages). No function here is "parity
unpinned".
"""
from . import attention, decode, fp8, layouts, merge, ring  # noqa: F401
