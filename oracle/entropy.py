"""Order-0 Huffman byte accounting of the stored codes (float-free, CPU).

Test infrastructure only -- see ``oracle/__init__.py``.

kvtc_cache page, module docstring "Byte accounting" and
``KVTCKVCache.entropy_coding_gain``: the stored size is the entropy-coded
payload plus its table plus the projection basis; ``pre_entropy_bytes`` is
the fixed-width size; the coder is an order-0 Huffman coder, and the
payload plus table never exceeds fixed-width packing (the coder falls back to
fixed width where Huffman does not pay for itself); the gain is
``pre_entropy_bytes / kvtc_bytes``, whose denominator carries the basis and
can therefore read below 1.  The pages do not print the coder itself; the
reading taken here (``_TensorKVTC._requantize`` hands the coder one code
array per surviving component together with its width):

* every kept component of a slot has its own order-0 Huffman code over the
  values that component takes across the slot's tokens;
* a code's table costs one byte per symbol of the component's alphabet
  (2^b code lengths describe a canonical Huffman code); a component with a
  single distinct value still spends one bit per token;
* a slot stores min(entropy-coded bytes, fixed-width bytes): the entropy-coded
  bytes are ceil(payload bits / 8) plus the tables, the fixed-width bytes the
  slot's packed rows.
"""
from __future__ import annotations

import heapq
import math

import numpy as np

__all__ = ["huffman_lengths", "component_bits", "slot_bytes", "layer_bytes"]


def huffman_lengths(counts):
    """Code length of each symbol of an order-0 Huffman code for ``counts``
    (symbols with count 0 get length 0).  One symbol in use: length 1."""
    counts = [int(c) for c in counts]
    used = [i for i, c in enumerate(counts) if c > 0]
    lengths = [0] * len(counts)
    if not used:
        return lengths
    if len(used) == 1:
        lengths[used[0]] = 1
        return lengths
    # heap of (weight, tie-break, symbols under the node); each merge adds one
    # bit to every symbol under the two merged nodes
    heap = [(counts[i], n, [i]) for n, i in enumerate(used)]
    heapq.heapify(heap)
    tie = len(heap)
    while len(heap) > 1:
        w1, _, s1 = heapq.heappop(heap)
        w2, _, s2 = heapq.heappop(heap)
        for i in s1 + s2:
            lengths[i] += 1
        heapq.heappush(heap, (w1 + w2, tie, s1 + s2))
        tie += 1
    return lengths


def component_bits(codes) -> int:
    """Payload bits of one component's code sequence under its own Huffman code."""
    codes = np.asarray(codes, dtype=np.int64)
    if codes.size == 0:
        return 0
    counts = np.bincount(codes)
    lengths = huffman_lengths(counts)
    return int(sum(int(c) * l for c, l in zip(counts, lengths)))


def slot_bytes(codes, bits):
    """One slot's codes [S, r] (components in index order, widths ``bits``):
    returns (fixed-width bytes, entropy-coded bytes, stored bytes)."""
    from .codec import row_bytes

    codes = np.asarray(codes)
    bits = np.asarray(bits)
    S = codes.shape[0]
    fixed = S * row_bytes(bits)
    payload = sum(component_bits(codes[:, k]) for k in range(len(bits)) if bits[k] > 0)
    table = sum(1 << int(b) for b in bits if b > 0)
    coded = (math.ceil(payload / 8) + table) if S else 0
    return fixed, coded, min(fixed, coded)


def layer_bytes(layer):
    """Totals over the slots of an ``OracleLayer`` in a coded mode: fixed-width
    payload, stored payload (after the fallback), the frozen parameter bytes and
    the gain fixed / (stored + parameters)."""
    from .codec import unpack_rows

    fixed = stored = 0
    for s in range(layer.n_slots):
        bits = layer.bits[layer.basis_of[s]]
        codes = unpack_rows(layer.rows[s], bits)
        f, _, st = slot_bytes(codes, bits)
        fixed += f
        stored += st
    params = layer.param_bytes()
    total = stored + params
    return {"pre_entropy": int(fixed), "stored_payload": int(stored), "params": int(params),
            "gain": (fixed / total) if total else 1.0}
