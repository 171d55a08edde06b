"""Sign-Muon sign extraction, 1-bit packing, majority vote and voted update.

Oracle module: test infrastructure only.

Passages followed ("Riepilogo Tecnico: SignMuon", §2):
* "Flusso Algoritmico" step 2: S = sign(U) elementwise, values in {-1, +1};
* step 3, all-gather variant: the signs are packed one bit per element and the
  packed buffers are all-gathered;
* "Meccanismo Principale" item 3 and step 4: the aggregate is the majority
  vote sign(sum_m S^(m)), computed locally by every worker, and the update is
  W <- W - eta * S_bar.

Readings where the pages are silent:
* tie rule: sign(0) = +1, so an element with U = +0 or -0 votes +1, and a vote
  whose sum is 0 (even number of workers, split evenly) gives +1; NaN is not
  below zero and also gives +1;
* packing: the matrix is flattened row-major (ignoring any leading-dimension
  padding); element j sits in bit (j mod 32) of uint32 word j // 32, bit 0 the
  least significant; unused bits of the last word are 0;
* the update W - lr*vote is one rounding in float32 (W's storage type); a
  bfloat16 W is updated in float32 and rounded to bf16 once.
"""
import numpy as np

from .bf16 import round_bf16


def sign(U):
    """Elementwise sign with sign(0) = +1 (and NaN -> +1), as float64 {-1,+1}."""
    U = np.asarray(U, dtype=np.float64)
    return np.where(U < 0, -1.0, 1.0)


def sign_bits(U):
    """Bit per element: 1 for a +1 sign, 0 for -1; row-major flattening."""
    return (~(np.asarray(U, dtype=np.float64) < 0)).astype(np.uint8).reshape(-1)


def num_words(numel):
    return (int(numel) + 31) // 32


def pack_bits(U):
    """Pack sign bits into uint32 words (little-endian bit order) with NumPy."""
    bits = sign_bits(U)
    nw = num_words(bits.size)
    padded = np.zeros(nw * 32, dtype=np.uint8)
    padded[: bits.size] = bits
    as_bytes = np.packbits(padded, bitorder="little")
    return as_bytes.view("<u4").astype(np.uint32)


def pack_bits_loop(U):
    """The same packing written as plain Python loops (small inputs only)."""
    flat = [float(v) for v in np.asarray(U, dtype=np.float64).reshape(-1)]
    words = [0] * num_words(len(flat))
    for j, v in enumerate(flat):
        if not (v < 0):
            words[j // 32] |= 1 << (j % 32)
    return np.array(words, dtype=np.uint32)


def unpack_bits(words, numel):
    """Bits of the first ``numel`` elements of packed uint32 words."""
    w = np.asarray(words, dtype="<u4")
    bits = np.unpackbits(w.view(np.uint8), bitorder="little")
    return bits[:numel]


def vote_counts(word_buffers, numel):
    """Number of workers voting +1 for each element."""
    c = np.zeros(int(numel), dtype=np.int64)
    for words in word_buffers:
        c += unpack_bits(words, numel)
    return c


def majority_vote(word_buffers, numel):
    """sign(sum_m S^(m)) with ties -> +1, from packed buffers, float64 {-1,+1}.

    With c workers voting +1 out of M, sum_m S = 2c - M, so the vote is +1 iff
    2c >= M.
    """
    M = len(word_buffers)
    c = vote_counts(word_buffers, numel)
    return np.where(2 * c >= M, 1.0, -1.0)


def sign_int8(U):
    """All-reduce variant payload ("Riepilogo Tecnico: SignMuon" §2 step 3,
    "Variante All-Reduce"; 8 bits per element, §2 "Efficienza di
    Comunicazione"): the sign of each element as int8 -1/+1, row-major,
    sign(0) = +1."""
    return np.where(np.asarray(U, dtype=np.float64).reshape(-1) < 0, -1, 1).astype(np.int8)


def int8_vote(sign_buffers):
    """Integer sum of the workers' int8 signs, then the local threshold
    sign(sum) with sign(0) = +1 (SignMuon §2 "Meccanismo Principale" item 3)."""
    total = np.zeros(np.asarray(sign_buffers[0]).size, dtype=np.int64)
    for s in sign_buffers:
        total += np.asarray(s, dtype=np.int64)
    return np.where(total >= 0, 1.0, -1.0)


def int8_vote_update(W, sign_buffers, lr, w_dtype="f32"):
    """W - lr * int8_vote(...), with the same float32 rounding as vote_update."""
    W = np.asarray(W)
    vote = int8_vote(sign_buffers).reshape(W.shape).astype(np.float32)
    new = (W.astype(np.float32) - np.float32(lr) * vote).astype(np.float64)
    if w_dtype == "bf16":
        new = round_bf16(new)
    return new


def vote_polar_update(W, word_buffers, lr, steps=5, a=3.4445, b=-4.7750, c=2.0315):
    """The optional local polar step (SignMuon §2 "Flusso Algoritmico" step
    5): the voted sign matrix S_bar is orthogonalised locally with the same
    Newton-Schulz iteration before the update, W <- W - lr * NS(S_bar).
    Returns float64 W (no storage rounding)."""
    from .muon import newton_schulz
    W = np.asarray(W, dtype=np.float64)
    S = majority_vote(word_buffers, W.size).reshape(W.shape)
    return W - lr * newton_schulz(S, steps, a, b, c)


def vote_update(W, word_buffers, lr, w_dtype="f32"):
    """W - lr * vote, one float32 rounding (then bf16 rounding for bf16 W).

    ``W`` holds the stored values (float32 or bf16 values as floats); the
    result has W's shape and is returned as float64 holding the stored values.
    """
    W = np.asarray(W)
    vote = majority_vote(word_buffers, W.size).reshape(W.shape).astype(np.float32)
    w32 = W.astype(np.float32)
    new = w32 - np.float32(lr) * vote            # float32 arithmetic, one rounding
    new = new.astype(np.float64)
    if w_dtype == "bf16":
        new = round_bf16(new)
    return new
