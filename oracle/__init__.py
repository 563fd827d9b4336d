"""CPU oracle for the OSCAR INT2 KV-cache hot path — TEST INFRASTRUCTURE ONLY.

A plain, slow, deliberately unoptimised restatement of what the path computes,
in float64 (and in explicit IEEE float32 where the quantizer's decisions are
made), written from the method's description and sharing no code with the CUDA
library.  Only the test suite, the smoke check and the benchmark's CPU-baseline
leg may import it; the product path never does.

Sources cited in this package:
  [Article]  "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化" (66bd.net
             overview article), sections "OSCAR 的动机" (Fig. 1) and
             "OSCAR 的设计" (Fig. 2).
  [Abstract] "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
             Cache Quantization" (arXiv 2605.17757 listing), Abstract and the
             Chinese summary "摘要".

Modules:
  rotation   R = U·H·P; Haar U from a Gaussian matrix; covariance-aligned U;
             calibration covariances Q^T Q and (SV)^T (SV).
  quant      exactly-rounded rotation, clip + asymmetric per-group INT2
             quantizer, 4-codes-per-byte packing, dequantization.
  attention  fp64 softmax attention, segment-wise online softmax + LSE merge,
             the three-segment decode.
  pool       the three-segment pool's bookkeeping: prefill, demote, append.
  accounting effective bits per KV element.

Parity status: every function here is pinned by tests/test_oracle_*.py
against closed forms, brute force (exact rationals) or library routines;
covariance-mode eigenvectors are pinned only where eigenvalues are distinct.
"""
