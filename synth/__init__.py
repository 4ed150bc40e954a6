"""Seeded synthetic inputs for cross-model KV-cache transfer.

This module is shared by the float64 oracle's tests, the GPU parity tests and
the benchmark.  It holds *random draws only*: Gaussian content with per-channel
log-normal scales, hidden layer selections, hidden affine weights and biases,
noise draws, ragged sequence lengths and position vectors.  It contains none of
the method's arithmetic (no RoPE, no feature concatenation, no affine map, no
statistics): composing draws into "stored" caches is done by whoever consumes
them (the oracle for small cases, the library's own apply call for benchmark
data).

Recipe (shapes and distributions of the pages' workloads; real captures and the
FineWeb-Edu calibration text are not available, these stand in for them):

* content c ~ N(0, 1) * s_ch with s_ch = exp(N(0, sigma^2)) drawn once per
  (layer, kv-head, dim) channel; sigma = 0.5 for the tiny pair, 1.0 otherwise;
* hidden selection: per target layer, k distinct source layers, ascending;
* hidden weights W ~ N(0, 1) / sqrt(k*H*d), stored [p][q] (inputs x outputs),
  bias b ~ N(0, 0.1^2);
* noise draws are standard normal; the consumer scales them (sigma = 1e-3, or
  per column to a signal-to-noise ratio);
* ragged batches: lengths uniform in [lo, hi], positions restart at 0 per
  sequence, sequences packed along the token axis;
* correlated layers (full-size solver checks): every layer of a cache is
  s_ch * (rho * z + sqrt(1 - rho^2) * e_l) with one shared draw z, so the
  channel marginals are unchanged and layers correlate by rho^2.
"""
from .generators import (  # noqa: F401
    channel_scales,
    content,
    hidden_selection,
    hidden_weights,
    noise,
    ragged_lengths,
    packed_positions,
    torch_content,
    torch_content_shared,
    torch_weights,
)
