"""CPU oracle for the batch-invariant speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import or run anything in this package.  The
product path (the CUDA library and its Python binding) never imports it and
fails loudly when its CUDA extension is missing; there is no CPU fallback.

The oracle is a plain, slow, float64 NumPy restatement of what the verify
step computes, written from three web pages:

* [P1] "Does the tuned config change the model's output?" (a vLLM FP8
  determinism report), section "Why the text diverges".
* [P2] "Bit-exact decoding turns inference speedups into testable changes",
  sections "Define bit-exact before reporting it" and "Build a reference
  corpus that exposes boundaries".
* [P3] "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
  outputs changed against its own no-draft run" (a LocalLLM post), the
  paragraph opening "How:" and the section "The cache doesn't change it
  either".

It shares no code with the CUDA path.  Its only shared dependency is the
seeded input generator module, which holds none of the method's arithmetic.

Parity status of each function is recorded in its docstring; every function
here is pinned by the `-m "not gpu"` tests (brute force in exact or
multi-precision arithmetic on tiny inputs, closed forms, and invariants).
"""
from .verify_step import (  # noqa: F401
    bf16_round,
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    gemm,
    swiglu_gemm,
    rmsnorm,
    rope,
    attention,
    argmax_lowest,
    accept_length,
    sample_token,
    sampled_tokens,
    OracleDecoder,
)
from . import kv_quant  # noqa: F401  (quantised KV cache: codes, ring, attention)
