"""Write tests/golden/blocks.json: one hand-chosen block per format.

Each block is packed from chosen field values (scales, mins, integer quants)
by the encoder below, written from the GGUF block convention that the pages
name ("Ntransformer", en.unwiki.net — About: Q4_0, Q8_0, Q4_K_M, Q5_K, Q6_K).
Expected element values are the closed forms applied to the chosen fields:

  Q8_0  v = d*q            Q4_0  v = d*(q-8)
  Q4_K  v = d*sc*q - dmin*m (q 4-bit)      Q5_K  same, q 5-bit
  Q6_K  v = d*sc*(q-32)

All chosen scales are powers of two or small integers, so every expected
value is exact in binary.  This script calls neither the oracle nor the CUDA
library; the oracle tests decode these bytes and must recover the fields and
values.  Run:  python tests/golden/make_golden.py
"""
import json
import os

HALF = {1.0: 0x3C00, 0.5: 0x3800, 2.0: 0x4000, 0.25: 0x3400}


def le16(v):
    return [v & 0xFF, v >> 8]


def q8_0():
    d = 0.5
    q = [i - 16 for i in range(32)]
    b = le16(HALF[d]) + [x & 0xFF for x in q]
    return dict(fmt="Q8_0", bytes=b, d=d, q=q, values=[d * x for x in q])


def q4_0():
    d = 2.0
    # element i < 16 in the low nibble of qs[i]; element i + 16 in its high nibble
    q = [i for i in range(16)] + [15 - i for i in range(16)]
    qs = [q[i] | (q[i + 16] << 4) for i in range(16)]
    b = le16(HALF[d]) + qs
    return dict(fmt="Q4_0", bytes=b, d=d, q=q, values=[d * (x - 8) for x in q])


SC = [1, 2, 3, 4, 17, 33, 50, 63]   # sub-block scales (6-bit), high bits exercised for j >= 4
MN = [0, 5, 10, 15, 20, 40, 48, 63]  # sub-block mins (6-bit)


def pack_scales12(sc, mn):
    """K-quant scales[12]: bytes 0-3 low 6 bits = sc[0..3], top 2 bits = sc[4..7] bits 4-5;
    bytes 4-7 the same for the mins; bytes 8-11 low nibble = sc[4..7] bits 0-3, high nibble =
    mn[4..7] bits 0-3."""
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | (((sc[j + 4] >> 4) & 3) << 6)
        s[j + 4] = (mn[j] & 63) | (((mn[j + 4] >> 4) & 3) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return s


def kq_nibbles():
    """q[256] 4-bit: sub-block j element l."""
    q = []
    for j in range(8):
        c = j // 2
        for l in range(32):
            q.append((l + c) % 16 if j % 2 == 0 else (3 * l + c) % 16)
    return q


def pack_qs128(q4):
    """qs[128]: chunk c = sub-blocks 2c (low nibbles) and 2c+1 (high nibbles)."""
    qs = []
    for c in range(4):
        for l in range(32):
            qs.append(q4[64 * c + l] | (q4[64 * c + 32 + l] << 4))
    return qs


def pack_q4_k(d_bits, dmin_bits, sc, mn, q):
    """Q4_K block bytes: d | dmin (f16 bits) | scales[12] | qs[128]; q[256] 4-bit."""
    return le16(d_bits) + le16(dmin_bits) + pack_scales12(sc, mn) + pack_qs128(q)


def pack_q5_k(d_bits, dmin_bits, sc, mn, q):
    """Q5_K block bytes: d | dmin | scales[12] | qh[32] | qs[128]; q[256] 5-bit, the fifth bit of
    element l of sub-block j is bit j of qh[l]."""
    qh = [0] * 32
    for i in range(256):
        qh[i % 32] |= ((q[i] >> 4) & 1) << (i // 32)
    return le16(d_bits) + le16(dmin_bits) + pack_scales12(sc, mn) + qh + pack_qs128([x & 15 for x in q])


def pack_q6_k(d_bits, sc, q):
    """Q6_K block bytes: ql[128] | qh[64] | scales[16] (int8) | d; q[256] 6-bit."""
    ql = [0] * 128
    qh = [0] * 64
    for h in range(2):
        for l in range(32):
            e0, e1, e2, e3 = (q[128 * h + l + 32 * g] for g in range(4))
            # ql[64h + l]: low nibble = element l, high nibble = element l + 64
            ql[64 * h + l] = (e0 & 15) | ((e2 & 15) << 4)
            # ql[64h + l + 32]: low nibble = element l + 32, high nibble = element l + 96
            ql[64 * h + l + 32] = (e1 & 15) | ((e3 & 15) << 4)
            # qh[32h + l]: bits 2g..2g+1 = top two bits of element l + 32g
            qh[32 * h + l] = (e0 >> 4) | ((e1 >> 4) << 2) | ((e2 >> 4) << 4) | ((e3 >> 4) << 6)
    return ql + qh + [x & 0xFF for x in sc] + le16(d_bits)


def q4_k():
    d, dmin = 1.0, 0.5
    q = kq_nibbles()
    b = pack_q4_k(HALF[d], HALF[dmin], SC, MN, q)
    vals = [d * SC[i // 32] * q[i] - dmin * MN[i // 32] for i in range(256)]
    return dict(fmt="Q4_K", bytes=b, d=d, dmin=dmin, sc=SC, m=MN, q=q, values=vals)


def q5_k():
    d, dmin = 1.0, 0.5
    lo = kq_nibbles()
    qh = [(l * 37 + 11) & 0xFF for l in range(32)]   # bit j of qh[l] = 5th bit of element l of sub-block j
    q = [lo[i] | (((qh[i % 32] >> (i // 32)) & 1) << 4) for i in range(256)]
    b = pack_q5_k(HALF[d], HALF[dmin], SC, MN, q)
    assert b[16:48] == qh
    vals = [d * SC[i // 32] * q[i] - dmin * MN[i // 32] for i in range(256)]
    return dict(fmt="Q5_K", bytes=b, d=d, dmin=dmin, sc=SC, m=MN, q=q, values=vals)


def q6_k():
    d = 0.25
    sc = [-128, -7, 0, 1, 5, 127, -1, 64, 2, -3, 9, -50, 33, 100, -100, 17]
    q = [(7 * i + (i // 16)) % 64 for i in range(256)]  # 6-bit quants
    b = pack_q6_k(HALF[d], sc, q)
    vals = [d * sc[(i // 128) * 8 + (i % 128) // 16] * (q[i] - 32) for i in range(256)]
    return dict(fmt="Q6_K", bytes=b, d=d, sc=sc, q=q, values=vals)


def main():
    blocks = [q8_0(), q4_0(), q4_k(), q5_k(), q6_k()]
    for blk in blocks:
        blk["hex"] = bytes(blk.pop("bytes")).hex()
    doc = {
        "source": "GGUF block convention for the formats named on 'Ntransformer' (en.unwiki.net), About; "
                  "fields chosen by hand, values = closed forms on the chosen fields",
        "blocks": blocks,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "blocks.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
