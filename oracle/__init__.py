"""Float64 CPU oracle of the projected-and-quantized KV cache hot path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import anything under ``oracle/``.  The
product package never does, and this package imports nothing from it: the
two share no code.

What it computes, step by step, in plain NumPy float64 (each function cites
the passage it follows; "kvtc_cache", "turboquant_cache" and "palu_cache"
name the three documentation pages of the VeloxQuant-MLX caches):

* ``fit``   -- local PCA by covariance eigendecomposition, the dynamic
  programming bit allocation (and its brute-force check), frozen uniform
  min/step, the PALU hi/lo bit split, Lloyd-Max centroids for a Gaussian and
  the seeded orthogonal rotation;
* ``codec`` -- projection, the three quantisers (uniform, per-token group
  scale, scalar codebook), the per-token int8 value quantiser, LSB-first
  bit packing into byte-aligned segments and reconstruction;
* ``layer`` -- a cache layer with the append / fetch / trim / nbytes
  semantics of the C ABI, built from the two modules above;
* ``attend`` -- decode attention of one query per (batch, query head) over
  the decoded keys and values of two layers (softmax of the scaled scores,
  weighted sum of the values);
* ``entropy`` -- order-0 Huffman byte accounting of the stored codes with
  the fixed-width fallback and the entropy-coding gain;
* ``prod`` -- the TurboQuantProd residual sketch (QJL sign bits and an fp16
  residual norm over the MSE stage) and the outlier two-stream key store,
  their decode, score estimate and attention.

Parity pins (tests/test_oracle_*.py) tie every function to something other
than itself: the bit layouts the turboquant_cache page prints, closed forms,
Max's 1960 table, brute force and invariants.  No function here is
"parity unpinned".
"""
from . import fit, codec, layer, attend, entropy, prod  # noqa: F401
