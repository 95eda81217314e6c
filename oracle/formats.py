"""Exact decoding of one expert's pageable bytes into float64 weight matrices.

Source: "Running an MoE Model Larger Than Your VRAM", section "What does Paged
Experts actually do?" (PR #42557 adds bf16, block-FP8 and GPTQ experts) and
section "Can paging change the model's outputs?" (every per-expert tensor,
including scales and zero points, is paged with the expert).

An expert is one contiguous byte string that holds all of its tensors. The
layout is this library's own (the pages fix none); it is restated here from the
layout contract, independently of the CUDA code:

  bf16  (format 0)
      W_gu  bf16 [2I][H]   rows 0..I-1 gate_proj, rows I..2I-1 up_proj
      W_d   bf16 [H][I]    down_proj
  block-FP8 (format 1), H and I multiples of 128
      Q_gu  e4m3 [2I][H]
      Q_d   e4m3 [H][I]
      S_gu  fp32 [2I/128][H/128]   one scale per 128x128 block: w = e4m3(q) * s
      S_d   fp32 [H/128][I/128]
  GPTQ int4, group 128 (format 2), H and I multiples of 128
      Q_gu  u8 [2I][H/2]   element c of a row: byte c//2, low nibble if c even
      Q_d   u8 [H][I/2]
      SZ_gu fp16 [2I][H/128][2]   (scale, zero) per output row and input group
      SZ_d  fp16 [H][I/128][2]
      w[n, c] = (q[n, c] - z[n, c//128]) * s[n, c//128]
  MXFP4 (format 3), H and I multiples of 128; the OCP microscaling layout: 32 inputs
  share one power-of-two scale
      Q_gu  u8 [2I][H/2]   FP4 E2M1 codes, element c of a row: byte c//2, low nibble if c even
      Q_d   u8 [H][I/2]
      X_gu  u8 [2I][H/32]  E8M0 scale per output row and block of 32 inputs
      X_d   u8 [H][I/32]
      w[n, c] = e2m1(q[n, c]) * 2^(X[n, c//32] - 127)
  NVFP4 (format 4), H and I multiples of 128; two-level scaling: 16 inputs share one
  e4m3 block scale, and each matrix has one fp32 tensor scale (gate_proj and up_proj,
  stored as one fused matrix, share theirs). The pages name NVFP4 among the formats of
  section "What does Paged Experts actually do?" (PR #45787) without its layout; this
  is the two-level encoding the name stands for.
      Q_gu  u8 [2I][H/2]   FP4 E2M1 codes, element c of a row: byte c//2, low nibble if c even
      Q_d   u8 [H][I/2]
      T_gu  fp32, then 12 bytes of padding
      B_gu  u8 [2I][H/16]  e4m3 block scale per output row and block of 16 inputs
      T_d   fp32, then 12 bytes of padding
      B_d   u8 [H][I/16]
      w[n, c] = e2m1(q[n, c]) * e4m3(B[n, c//16]) * T

All sections are packed back to back in the order listed, with no other padding.
TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

import numpy as np

BF16, FP8_BLOCK128, INT4_GPTQ_G128, MXFP4, NVFP4 = 0, 1, 2, 3, 4


def expert_nbytes(fmt, H, I):
    """Bytes of one expert in the given format (sum of the sections above)."""
    n_w = 3 * H * I
    if fmt == BF16:
        return 2 * n_w
    if fmt == FP8_BLOCK128:
        return n_w + 4 * ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128))
    if fmt == INT4_GPTQ_G128:
        return n_w // 2 + 4 * ((2 * I) * (H // 128) + H * (I // 128))
    if fmt == MXFP4:
        return n_w // 2 + (2 * I) * (H // 32) + H * (I // 32)
    if fmt == NVFP4:
        return n_w // 2 + 16 + (2 * I) * (H // 16) + 16 + H * (I // 16)
    raise ValueError("unknown format")


def bf16_bits_to_f64(u16):
    """bf16 bit patterns -> float64 (exact: bf16 is the top half of an fp32)."""
    u32 = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def e4m3_value(code):
    """Value of one OCP FP8 E4M3 ("e4m3fn") code, from the format's definition.

    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
    subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
    """
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e2m1_value(code):
    """Value of one FP4 E2M1 code (the OCP microscaling element type), from its fields.

    1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent 0 is subnormal
    (m/2); there is no infinity or NaN.
    """
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * (m / 2.0)
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def e8m0_value(byte):
    """Value of one E8M0 scale: 2^(byte - 127); 0xFF is NaN."""
    return float("nan") if byte == 0xFF else 2.0 ** (int(byte) - 127)


E8M0_TABLE = np.array([e8m0_value(b) for b in range(256)], dtype=np.float64)


def _take(buf, off, nbytes):
    return buf[off:off + nbytes], off + nbytes


def decode_expert(buf, fmt, H, I):
    """Decode one expert's bytes -> (W_g [I,H], W_u [I,H], W_d [H,I]) float64."""
    buf = np.frombuffer(bytes(buf), dtype=np.uint8) if not isinstance(buf, np.ndarray) else buf.view(np.uint8).reshape(-1)
    if buf.size != expert_nbytes(fmt, H, I):
        raise ValueError("expert byte size does not match the format")
    off = 0
    if fmt == BF16:
        raw, off = _take(buf, off, 2 * 2 * I * H)
        Wgu = bf16_bits_to_f64(raw.view(np.uint16)).reshape(2 * I, H)
        raw, off = _take(buf, off, 2 * H * I)
        Wd = bf16_bits_to_f64(raw.view(np.uint16)).reshape(H, I)
    elif fmt == FP8_BLOCK128:
        qgu, off = _take(buf, off, 2 * I * H)
        qd, off = _take(buf, off, H * I)
        sgu, off = _take(buf, off, 4 * (2 * I // 128) * (H // 128))
        sd, off = _take(buf, off, 4 * (H // 128) * (I // 128))
        Sgu = sgu.view(np.float32).astype(np.float64).reshape(2 * I // 128, H // 128)
        Sd = sd.view(np.float32).astype(np.float64).reshape(H // 128, I // 128)
        Wgu = E4M3_TABLE[qgu].reshape(2 * I, H)
        Wd = E4M3_TABLE[qd].reshape(H, I)
        # block (n // 128, c // 128) carries one scale
        Wgu = Wgu * np.repeat(np.repeat(Sgu, 128, axis=0), 128, axis=1)
        Wd = Wd * np.repeat(np.repeat(Sd, 128, axis=0), 128, axis=1)
    elif fmt == INT4_GPTQ_G128:
        qgu, off = _take(buf, off, I * H)
        qd, off = _take(buf, off, H * I // 2)
        szgu, off = _take(buf, off, 4 * 2 * I * (H // 128))
        szd, off = _take(buf, off, 4 * H * (I // 128))
        Wgu = _int4_rows(qgu, szgu, 2 * I, H)
        Wd = _int4_rows(qd, szd, H, I)
    elif fmt == MXFP4:
        qgu, off = _take(buf, off, I * H)
        qd, off = _take(buf, off, H * I // 2)
        xgu, off = _take(buf, off, 2 * I * (H // 32))
        xd, off = _take(buf, off, H * (I // 32))
        Wgu = _mxfp4_rows(qgu, xgu, 2 * I, H)
        Wd = _mxfp4_rows(qd, xd, H, I)
    elif fmt == NVFP4:
        qgu, off = _take(buf, off, I * H)
        qd, off = _take(buf, off, H * I // 2)
        tgu, off = _take(buf, off, 16)
        bgu, off = _take(buf, off, 2 * I * (H // 16))
        td, off = _take(buf, off, 16)
        bd, off = _take(buf, off, H * (I // 16))
        Wgu = _nvfp4_rows(qgu, bgu, tgu, 2 * I, H)
        Wd = _nvfp4_rows(qd, bd, td, H, I)
    else:
        raise ValueError("unknown format")
    if off != buf.size:
        raise AssertionError("layout sections do not cover the expert")
    return Wgu[:I], Wgu[I:], Wd


def _int4_rows(qbytes, szbytes, n_rows, n_cols):
    """GPTQ int4 rows: q nibbles (low first), per-(row, group of 128) fp16 (s, z)."""
    q = qbytes.reshape(n_rows, n_cols // 2)
    nib = np.empty((n_rows, n_cols), dtype=np.float64)
    nib[:, 0::2] = (q & 0x0F).astype(np.float64)
    nib[:, 1::2] = (q >> 4).astype(np.float64)
    sz = szbytes.view(np.float16).astype(np.float64).reshape(n_rows, n_cols // 128, 2)
    s = np.repeat(sz[:, :, 0], 128, axis=1)
    z = np.repeat(sz[:, :, 1], 128, axis=1)
    return (nib - z) * s


def _mxfp4_rows(qbytes, xbytes, n_rows, n_cols):
    """MXFP4 rows: E2M1 nibbles (low first), one E8M0 scale per (row, block of 32)."""
    q = qbytes.reshape(n_rows, n_cols // 2)
    codes = np.empty((n_rows, n_cols), dtype=np.uint8)
    codes[:, 0::2] = q & 0x0F
    codes[:, 1::2] = q >> 4
    x = E8M0_TABLE[xbytes.reshape(n_rows, n_cols // 32)]
    return E2M1_TABLE[codes] * np.repeat(x, 32, axis=1)


def _nvfp4_rows(qbytes, bbytes, tbytes, n_rows, n_cols):
    """NVFP4 rows: E2M1 nibbles (low first), one e4m3 scale per (row, block of 16), and
    the matrix's fp32 tensor scale (the first 4 of its 16 bytes)."""
    q = qbytes.reshape(n_rows, n_cols // 2)
    codes = np.empty((n_rows, n_cols), dtype=np.uint8)
    codes[:, 0::2] = q & 0x0F
    codes[:, 1::2] = q >> 4
    b = E4M3_TABLE[bbytes.reshape(n_rows, n_cols // 16)]
    t = float(tbytes[:4].view(np.float32)[0])
    return E2M1_TABLE[codes] * np.repeat(b, 16, axis=1) * t
