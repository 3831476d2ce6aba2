"""CPU oracle for causal prefill attention with per-block FP8 quantisation.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
benchmark's CPU-baseline arm may import this package. The product path never
calls it: it has no CPU fallback, and the CUDA library shares no code, header,
table or constant with this package.

What it computes, and the passages it follows:

* ``fp8.e4m3_rne`` / ``fp8.e4m3_decode`` -- the e4m3 ("fn" variant, bias 7,
  largest finite 448) format and round-to-nearest-even, from "FP8 GEMM on
  CDNA4" section 2.1 (format table) and section 2.3 (RNE), and the e4m3 facts
  in "ZYFA: Fast and Accurate FP8 Attention on AMD MI355X" (section
  "Precision and Underflow of FP8 Probabilities" and footnote 7).
* ``fp8.quantize_fp8`` -- per-block amax, scale = amax / 448 with a guard for
  all-zero blocks, code = RNE(x / scale): "FP8 GEMM on CDNA4" section 2.2,
  with per-(batch, head, 128-token block) granularity. The optional
  128-point Walsh-Hadamard rotation of Q and K comes from the ZYFA post,
  section "FP8 Error in Full-Model Inference" and footnote 2.
* ``attention.causal_attention`` -- exact softmax attention with a causal
  mask in float64, the computation the ZYFA kernels perform ("Introduction":
  causal forward attention; "Methodology and Limitations": equal query and
  key lengths), with grouped-query heads.
* ``attention.causal_attention_prefix`` -- the same definition for queries
  that continue a cached prefix (query i at position P + i sees keys
  0 .. P + i); the pages list paged caches as future work ("Methodology and
  Limitations").

Every function is pinned by ``tests/test_oracle_*.py`` against facts that do
not come from this package: printed e4m3 codes, torch's float8 cast, SciPy's
Hadamard matrix, PyTorch's float64 scaled-dot-product attention, brute force
on tiny inputs and closed forms.
"""
from . import fp8, attention  # noqa: F401
