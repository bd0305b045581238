"""Byte layout of one paged INT2 block, as a (token, channel) -> (byte, bit) map.

Oracle; test infrastructure only.  Written from the layout specification in
the library's public header documentation (the packed-block description),
not from the CUDA code.

[IT] "Architettura del Sistema di Serving": a paged, mixed-precision cache;
[ES] §2.2 B: the INT2 history is stored in a paged cache after the fixed
rotation and clipping.  The pages give no bit layout; this one is ours.

One block holds one page (64 consecutive positions) of one KV head:

    bytes [   0, 2048)  K codes   (64 tokens x 128 channels x 2 bits)
    bytes [2048, 2304)  K scales  fp16 [64 tokens][2 groups], little endian
    bytes [2304, 4352)  V codes
    bytes [4352, 4608)  V scales  fp16 [64 tokens][2 groups]

Codes are grouped in 16-token tiles of 512 bytes (tile T = t // 16 starts at
byte 512 T of the code area).  Inside a tile, with u = t % 16, the 2-bit code
of rotated channel j sits at

    K:  lane  = 4 (u % 8) + (j // 4) % 4
        word  = 2 (u // 8) + j // 64
        bit   = 8 (j % 4) + 2 (2 ((j // 32) % 2) + (j // 16) % 2)
    V:  lane  = 4 (j % 8) + (u % 8) // 2
        word  = 2 (u // 8) + (j % 16) // 8
        bit   = 16 (u % 2) + 2 (j // 16)

    byte offset = 512 T + 16 lane + 4 word + bit // 8,   bit-in-byte = bit % 8.

Each (tile, lane, word) is a little-endian 32-bit word.  A K token owns whole
32-bit words and a V token owns whole 16-bit halves, so tokens never share a
byte.
"""

import numpy as np

PAGE_TOKENS = 64
HEAD_DIM = 128
GROUP = 64
CODE_BYTES = 2048
SCALE_BYTES = 256
K_CODES = 0
K_SCALES = 2048
V_CODES = 2304
V_SCALES = 4352
BLOCK_BYTES = 4608


def k_code_position(t, j):
    """(byte, bit-in-byte) of the K code of token t (0..63), channel j (0..127)."""
    T, u = divmod(t, 16)
    lane = 4 * (u % 8) + (j // 4) % 4
    word = 2 * (u // 8) + j // 64
    bit = 8 * (j % 4) + 2 * (2 * ((j // 32) % 2) + (j // 16) % 2)
    return 512 * T + 16 * lane + 4 * word + bit // 8, bit % 8


def v_code_position(t, j):
    """(byte, bit-in-byte) of the V code of token t (0..63), channel j (0..127)."""
    T, u = divmod(t, 16)
    lane = 4 * (j % 8) + (u % 8) // 2
    word = 2 * (u // 8) + (j % 16) // 8
    bit = 16 * (u % 2) + 2 * (j // 16)
    return 512 * T + 16 * lane + 4 * word + bit // 8, bit % 8


def _position_tables():
    kb = np.zeros((PAGE_TOKENS, HEAD_DIM), dtype=np.int64)
    ki = np.zeros_like(kb)
    vb = np.zeros_like(kb)
    vi = np.zeros_like(kb)
    for t in range(PAGE_TOKENS):
        for j in range(HEAD_DIM):
            kb[t, j], ki[t, j] = k_code_position(t, j)
            vb[t, j], vi[t, j] = v_code_position(t, j)
    return kb, ki, vb, vi


_TABLES = None


def _tables():
    global _TABLES
    if _TABLES is None:
        _TABLES = _position_tables()
    return _TABLES


def _pack_codes(codes, byte_idx, bit_idx):
    area = np.zeros(CODE_BYTES, dtype=np.uint8)
    for t in range(codes.shape[0]):
        for j in range(HEAD_DIM):
            area[byte_idx[t, j]] |= np.uint8((int(codes[t, j]) & 3) << int(bit_idx[t, j]))
    return area


def _unpack_codes(area, byte_idx, bit_idx, n_tokens=PAGE_TOKENS):
    area = np.asarray(area, dtype=np.uint8)
    return ((area[byte_idx[:n_tokens]] >> bit_idx[:n_tokens].astype(np.uint8)) & 3).astype(np.uint8)


def pack_block(k_codes, k_scales, v_codes, v_scales):
    """Assemble one 4608-byte block from codes [n, 128] and fp16-valued scales [n, 2].

    Rows n < 64 fill the first n token rows; the rest stay zero.
    """
    kb, ki, vb, vi = _tables()
    n = np.asarray(k_codes).shape[0]
    block = np.zeros(BLOCK_BYTES, dtype=np.uint8)
    block[K_CODES:K_CODES + CODE_BYTES] = _pack_codes(np.asarray(k_codes), kb, ki)
    block[V_CODES:V_CODES + CODE_BYTES] = _pack_codes(np.asarray(v_codes), vb, vi)
    ks = np.zeros((PAGE_TOKENS, 2), dtype=np.float16)
    vs = np.zeros((PAGE_TOKENS, 2), dtype=np.float16)
    ks[:n] = np.asarray(k_scales, dtype=np.float64).astype(np.float16)
    vs[:n] = np.asarray(v_scales, dtype=np.float64).astype(np.float16)
    block[K_SCALES:K_SCALES + SCALE_BYTES] = ks.astype('<f2').view(np.uint8).reshape(-1)
    block[V_SCALES:V_SCALES + SCALE_BYTES] = vs.astype('<f2').view(np.uint8).reshape(-1)
    return block


def unpack_block(block, n_tokens=PAGE_TOKENS):
    """Inverse of pack_block: (k_codes, k_scales, v_codes, v_scales) for the first n tokens."""
    kb, ki, vb, vi = _tables()
    block = np.asarray(block, dtype=np.uint8).reshape(-1)
    if block.size != BLOCK_BYTES:
        raise ValueError("a block is %d bytes" % BLOCK_BYTES)
    kc = _unpack_codes(block[K_CODES:K_CODES + CODE_BYTES], kb, ki, n_tokens)
    vc = _unpack_codes(block[V_CODES:V_CODES + CODE_BYTES], vb, vi, n_tokens)
    ks = block[K_SCALES:K_SCALES + SCALE_BYTES].copy().view('<f2').reshape(PAGE_TOKENS, 2)
    vs = block[V_SCALES:V_SCALES + SCALE_BYTES].copy().view('<f2').reshape(PAGE_TOKENS, 2)
    return kc, ks[:n_tokens].astype(np.float64), vc, vs[:n_tokens].astype(np.float64)


def unpack_blocks(blocks):
    """Vectorised unpack_block over blocks [N, 4608] -> (kc [N,64,128], ks [N,64,2], vc, vs)."""
    kb, ki, vb, vi = _tables()
    blocks = np.asarray(blocks, dtype=np.uint8).reshape(-1, BLOCK_BYTES)
    kc = (blocks[:, K_CODES + kb] >> ki.astype(np.uint8)) & 3
    vc = (blocks[:, V_CODES + vb] >> vi.astype(np.uint8)) & 3
    ks = blocks[:, K_SCALES:K_SCALES + SCALE_BYTES].copy().view('<f2').reshape(-1, PAGE_TOKENS, 2)
    vs = blocks[:, V_SCALES:V_SCALES + SCALE_BYTES].copy().view('<f2').reshape(-1, PAGE_TOKENS, 2)
    return kc.astype(np.uint8), ks.astype(np.float64), vc.astype(np.uint8), vs.astype(np.float64)
