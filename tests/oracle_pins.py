"""Pins of the CPU oracle to facts outside itself.

Each check compares the oracle with something it does not compute itself:
values printed on the pages (tests/golden), hand-worked blocks, a library
routine (torch's float8_e4m3fn and numpy's float16 decoders), or exact
brute force on inputs whose sums are exact in fp64.  ``pin_failures(L)``
returns the list of failed checks for an oracle library ``L`` (``None`` = the
real oracle); the tests require it to be empty for the real oracle and
non-empty for every deliberately broken copy.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from golden_io import lines

DUAL, FAST = oracle.DUAL, oracle.FAST


def golden_codebook():
    rows = list(lines("codebook10.txt"))
    table = [int(v) for v in rows[0].split()]
    e2m1 = [float(v) for v in rows[1].split(":")[1].split()]
    return table, e2m1


def golden_layout():
    out = {}
    for ln in lines("block_layout.txt"):
        name, wpb, qs, sc, bb, bpw = ln.split()
        out[name] = (int(wpb), int(qs), int(sc), int(bb), float(bpw))
    return out


def golden_ue4m3():
    out = []
    for ln in lines("ue4m3_spot.txt"):
        b, e, m, v, hs, fin = ln.split()
        out.append((int(b, 16), int(e), int(m), float(v), float(hs), bool(int(fin))))
    return out


def golden_decoded_block():
    rows = list(lines("decoded_block.txt"))
    blk = np.array([int(v, 16) for v in rows[0].split()], dtype=np.uint8)
    w = np.array([float(v) for v in rows[1].split()] + [float(v) for v in rows[2].split()])
    return blk, w


def golden_hand_blocks():
    out = []
    for ln in lines("hand_blocks.txt"):
        name, var, qs, e0, e1, xa, xb, y, y_alt = ln.split()
        out.append(dict(name=name, variant=DUAL if var == "dual" else FAST, qs=int(qs, 16),
                        e0=int(e0, 16), e1=None if e1 == "-" else int(e1, 16),
                        xa=float(xa), xb=float(xb), y=float(y), y_alt=float(y_alt)))
    return out


def f16_bits(values) -> np.ndarray:
    return np.asarray(values, dtype=np.float16).view(np.uint16)


def hand_block_bytes(case) -> np.ndarray:
    blk = [case["qs"]] * 16 + [case["e0"]]
    if case["variant"] == DUAL:
        blk.append(case["e1"])
    return np.array(blk, dtype=np.uint8)


def torch_e4m3_values() -> np.ndarray:
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_failures(L=None) -> list[str]:
    fails: list[str] = []

    def check(name, ok):
        if not ok:
            fails.append(name)

    for section in (_pin_tables, _pin_scales, _pin_blocks, _pin_activations, _pin_brute_force,
                    _pin_validate, _pin_gate_up, _pin_attention, _pin_quantize):
        try:
            with np.errstate(invalid="ignore"):
                section(check, L)
        except Exception as exc:  # a broken oracle may also fail loudly
            fails.append(f"{section.__name__}: {type(exc).__name__}: {exc}")
    return fails


def _pin_tables(check, L):
    # 1. Codebook10 as printed; it is doubled E2M1 with 12 retuned to 10.
    table, e2m1 = golden_codebook()
    cb = [oracle.codebook(q, L) for q in range(16)]
    check("codebook table", cb == table)
    doubled = [2 * v for v in e2m1] + [-2 * v for v in e2m1]
    check("codebook vs doubled e2m1", all(
        (c == d) or (q % 8 == 7 and abs(d) == 12 and abs(c) == 10) for q, (c, d) in enumerate(zip(cb, doubled))))

    # 2. Block sizes and bits per weight as printed.
    lay = golden_layout()
    for name, var in (("dual", DUAL), ("fast", FAST)):
        wpb, qs, sc, bb, bpw = lay[name]
        got = oracle.block_bytes(var, L)
        check(f"block bytes {name}", got == bb == qs + sc)
        check(f"bpw {name}", abs(got * 8 / wpb - bpw) < 1e-12)


def _pin_scales(check, L):
    # 3. Scale decode: E4M3 value of every finite code equals torch's
    #    float8_e4m3fn decoder; spot values worked by hand; finiteness.
    ref = torch_e4m3_values()
    for s in range(0x7F):
        check(f"ue4m3 {s:#04x} vs torch", oracle.ue4m3(s, L) == ref[s])
        check(f"halfscale {s:#04x}", oracle.halfscale(s, L) == 0.5 * ref[s])
    for s in range(256):
        finite = s < 0x80 and np.isfinite(ref[s])
        check(f"validity {s:#04x}", oracle.scale_is_valid(s, L) == finite)
    for b, e, m, v, hs, fin in golden_ue4m3():
        check(f"spot validity {b:#04x}", oracle.scale_is_valid(b, L) == fin)
        if fin:
            check(f"spot value {b:#04x}", oracle.ue4m3(b, L) == v and oracle.halfscale(b, L) == hs)


def _pin_blocks(check, L):
    # 4. A block decoded by hand, weight by weight (signs, both halves, code 8 -> +0).
    blk, w_ref = golden_decoded_block()
    w = oracle.decode_block(blk, DUAL, L)
    check("decoded block", np.array_equal(w, w_ref) and not np.any(np.signbit(w[w == 0])))
    wd = oracle.dequant(blk, 1, 32, DUAL, L)[0]
    check("dequant = decode_block", np.array_equal(wd, w_ref))

    # 5. Single-block products worked by hand.
    for case in golden_hand_blocks():
        x = f16_bits([case["xa"]] * 16 + [case["xb"]] * 16)
        y = oracle.gemv(hand_block_bytes(case), x, 1, 32, case["variant"], L=L)[0]
        check(f"hand block {case['name']}", y == case["y"])


def _pin_activations(check, L):
    # 6. Activation decoders: every 7th fp16 / bf16 bit pattern vs numpy.
    bits = np.arange(65536, dtype=np.uint16)
    f16 = bits.view(np.float16).astype(np.float64)
    f16_o = np.array([oracle.act_value(b, oracle.ACT_F16, L) for b in range(0, 65536, 7)])
    check("fp16 decode", np.array_equal(f16_o, f16[::7], equal_nan=True))
    bf16 = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    bf16_o = np.array([oracle.act_value(b, oracle.ACT_BF16, L) for b in range(0, 65536, 7)])
    check("bf16 decode", np.array_equal(bf16_o, bf16[::7], equal_nan=True))


def _pin_brute_force(check, L):
    # 7. Brute force: x and weights chosen so every sum is exact in fp64, so
    #    the oracle must equal a dense numpy matmul of the dequantised matrix
    #    to the last bit (M > 1 and N > 1 catch swapped or transposed indices).
    rng = np.random.default_rng(7)
    for var in (DUAL, FAST):
        N, K, M = 5, 96, 3
        W = synth.weights(N, K, var, seed=3, stream=11)
        X = f16_bits(rng.integers(-8, 9, size=(M, K)).astype(np.float64) * 0.25)
        dense = oracle.dequant(W, N, K, var, L)
        Xf = X.view(np.float16).astype(np.float64)
        Y = oracle.gemm(W, X, N, K, var, nthreads=2, L=L)
        check(f"brute force exact {var}", np.array_equal(Y, Xf @ dense.T))
        # dense rows agree with block-by-block decoding
        rb = oracle.row_bytes(K, var, L)
        bb = oracle.block_bytes(var, L)
        blocks = np.concatenate([oracle.decode_block(W[n, b * bb:(b + 1) * bb], var, L)
                                 for n in range(N) for b in range(rb // bb)])
        check(f"dequant rows {var}", np.array_equal(blocks.reshape(N, K), dense))


def _pin_validate(check, L):
    # 8. Validation finds a planted non-finite scale byte (second half too).
    for var, off in ((DUAL, 16), (DUAL, 17), (FAST, 16)):
        N, K = 3, 64
        W = synth.weights(N, K, var, seed=0, stream=2).copy()
        bb = oracle.block_bytes(var, L)
        check(f"validate clean {var}", oracle.validate(W, N, K, var, L) == -1)
        flat = W.reshape(-1)
        flat[4 * bb + off] = 0x7F
        flat[5 * bb + 16] = 0x80
        check(f"validate planted {var}/{off}", oracle.validate(W, N, K, var, L) == 4)


def _gate_up_matrix(g_codes, u_codes, var):
    """2 x 32 rows (one gate row, one up row), half-scales 1.0: weight j of a
    row is Codebook10[code j] (codes for j < 16 only, the other half zero)."""
    W = np.zeros((2, synth.block_bytes(var)), dtype=np.uint8)
    for r, codes in enumerate((g_codes, u_codes)):
        for j, q in enumerate(codes):
            W[r, j] = q & 0xF
    W[:, 16:] = 0x40  # E4M3 2.0: half-scale 1.0
    return W


def _pin_gate_up(check, L):
    # 9. The fused gate/up product, reading R11: y = SiLU(g) * u with the gate
    #    rows first.  Pinned by identities of the logistic function, not by
    #    its formula: with u = 1,
    #      y(g) - y(-g) = g            (SiLU(g) = g * s(g), s(g) + s(-g) = 1)
    #      y(g) + y(-g) = g tanh(g/2)  (s(g) - s(-g) = tanh(g/2))
    #    The second identity holds for the logistic s only (not for the
    #    Gaussian CDF of GELU, nor for a sign-flipped exponent).
    for var in (DUAL, FAST):
        x = f16_bits(np.ones(32))
        # one gate weight 2 (code 2) and up weights summing to 3 (code 3): y = 3 SiLU(2)
        W = _gate_up_matrix([2], [3], var)
        y = oracle.gemv_gate_up(W, x, 1, 32, var, L=L)[0, 0]
        check(f"gate/up order {var}", abs(y - 3.0 * (1.0 + np.tanh(1.0))) < 1e-13)
        # identities over gate sums g = -20 .. 20 in steps of 0.5 (x scales the code-1 weight)
        gs = np.arange(-40, 41) * 0.5
        W = _gate_up_matrix([1], [1], var)
        odd, even = True, True
        for g in gs[gs > 0]:
            xp = f16_bits(np.r_[g, np.zeros(31)])
            xn = f16_bits(np.r_[-g, np.zeros(31)])
            # up row weight 1 * x = g as well, so divide it out: y / g = SiLU(+-g) / (+-g) * ...
            yp = oracle.gemv_gate_up(W, xp, 1, 32, var, L=L)[0, 0] / g
            yn = oracle.gemv_gate_up(W, xn, 1, 32, var, L=L)[0, 0] / -g
            odd &= abs((yp - yn) - g) <= 1e-12 * max(1.0, g)
            even &= abs((yp + yn) - g * np.tanh(g / 2)) <= 1e-12 * max(1.0, g)
        check(f"gate/up odd part {var}", odd)
        check(f"gate/up logistic even part {var}", even)
        # saturation: SiLU(30) = 30 to 1e-12, SiLU(-30) ~ -3e-12
        xp = f16_bits(np.r_[30.0, np.zeros(31)])
        xn = f16_bits(np.r_[-30.0, np.zeros(31)])
        yp = oracle.gemv_gate_up(W, xp, 1, 32, var, L=L)[0, 0]
        yn = oracle.gemv_gate_up(W, xn, 1, 32, var, L=L)[0, 0]
        check(f"gate/up saturation {var}", abs(yp / 900.0 - 1.0) < 1e-11 and abs(yn) < 1e-9)
    # brute force: random blocks, M > 1 and I > 1, every sum exact in fp64;
    # expected value through the tanh form of the identities above
    rng = np.random.default_rng(8)
    for var in (DUAL, FAST):
        I, K, M = 3, 96, 2
        W = synth.weights(2 * I, K, var, seed=4, stream=12)
        X = f16_bits(rng.integers(-8, 9, size=(M, K)).astype(np.float64) * 0.25)
        dense = oracle.dequant(W, 2 * I, K, var, L)
        Xf = X.view(np.float16).astype(np.float64)
        G, U = Xf @ dense[:I].T, Xf @ dense[I:].T
        want = 0.5 * G * (1.0 + np.tanh(G / 2)) * U
        got = oracle.gemv_gate_up(W, X, I, K, var, nthreads=2, L=L)
        check(f"gate/up brute force {var}", got.shape == (M, I) and np.allclose(got, want, rtol=1e-13, atol=1e-13))


def _kv_rows(codes, var, scale_byte=0x40):
    """Cache rows of D = 32 (one block each) from per-row code lists (weight j <
    16 = Codebook10[code j]; the rest 0), half-scales 1.0 by default."""
    bb = synth.block_bytes(var)
    R = np.zeros((len(codes), bb), dtype=np.uint8)
    for r, cs in enumerate(codes):
        for j, q in enumerate(cs):
            R[r, j] = q & 0xF
        R[r, 16:] = scale_byte
    return R


def _pin_attention(check, L):
    # 10. Decode attention over a ROCmFP4 K/V cache, reading R12.
    for var in (DUAL, FAST):
        D = 32
        dense = lambda R: oracle.dequant(R, R.shape[0], D, var, L)
        rng = np.random.default_rng(9)
        # (a) one token: the output is its V row exactly, whatever q
        K1 = _kv_rows([[3, 5, 9]], var)
        V1 = synth.weights(1, D, var, seed=5, stream=13)
        q = f16_bits(rng.integers(-4, 5, size=D) * 0.5)
        out = oracle.decode_attention(q, K1, V1, [1], 1, 1, 1, D, 1, 0.25, var, L=L)
        check(f"attn one token {var}", np.array_equal(out[0, 0], dense(V1)[0]))
        # (b) equal keys: the mean of the V rows
        T = 6
        Kc = np.repeat(_kv_rows([[1, 2, 3, 4]], var), T, axis=0)
        Vc = synth.weights(T, D, var, seed=5, stream=14)
        out = oracle.decode_attention(q, Kc, Vc, [T], 1, 1, 1, D, T, 0.3, var, L=L)
        check(f"attn equal keys {var}", np.allclose(out[0, 0], dense(Vc).mean(axis=0), rtol=1e-14, atol=1e-14))
        # (c) a dominant key, even at huge scores (max subtracted before exp)
        Kc = _kv_rows([[0], [7], [0], [0]], var)  # row 1: weight 0 = 10
        qd = f16_bits(np.r_[64.0, np.zeros(D - 1)])  # score of row 1: 640 * scale
        Vc = synth.weights(4, D, var, seed=5, stream=15)
        out = oracle.decode_attention(qd, Kc, Vc, [4], 1, 1, 1, D, 4, 4.0, var, L=L)
        check(f"attn dominant key {var}", np.all(np.isfinite(out)) and np.allclose(out[0, 0], dense(Vc)[1], rtol=1e-15, atol=1e-15))
        # (d) two tokens: p0 = (1 + tanh((s0 - s1)/2)) / 2 with s1 = 0
        Kc = _kv_rows([[1], [0]], var)  # s0 = scale * q[0]
        q2 = f16_bits(np.r_[3.0, np.zeros(D - 1)])
        Vc = synth.weights(2, D, var, seed=5, stream=16)
        out = oracle.decode_attention(q2, Kc, Vc, [2], 1, 1, 1, D, 2, 0.5, var, L=L)
        p0 = 0.5 * (1.0 + np.tanh(0.5 * 1.5))
        Vd = dense(Vc)
        check(f"attn two tokens {var}", np.allclose(out[0, 0], p0 * Vd[0] + (1 - p0) * Vd[1], rtol=1e-14, atol=1e-14))
        # (e) grouped heads: H = 4 over Hkv = 2, one token each: head h reads KV head h // 2
        Kc = _kv_rows([[1], [2]], var)
        Vc = synth.weights(2, D, var, seed=5, stream=17)
        q4 = f16_bits(rng.integers(-4, 5, size=(4, D)) * 0.5)
        out = oracle.decode_attention(q4, Kc, Vc, [1], 1, 4, 2, D, 1, 0.25, var, L=L)
        Vd = dense(Vc)
        check(f"attn grouped heads {var}", all(np.array_equal(out[0, h], Vd[h // 2]) for h in range(4)))
        # (f) lengths: rows past lens[b] are ignored, lens 0 gives zeros (B = 2, Tmax = 4)
        Kc = synth.weights(8, D, var, seed=5, stream=18)
        Vc = synth.weights(8, D, var, seed=5, stream=19)
        qb = f16_bits(rng.integers(-4, 5, size=(2, D)) * 0.25)
        out = oracle.decode_attention(qb, Kc, Vc, [3, 0], 2, 1, 1, D, 4, 0.2, var, L=L)
        K2, V2 = Kc.copy(), Vc.copy()
        K2[3] ^= 0x33
        V2[3] ^= 0x55
        out2 = oracle.decode_attention(qb, K2, V2, [3, 0], 2, 1, 1, D, 4, 0.2, var, L=L)
        check(f"attn lengths {var}", np.array_equal(out, out2) and np.all(out[1] == 0) and np.any(out[0] != 0))
        # (g) scale: a power-of-two scale equals that scaling of q (exact)
        o1 = oracle.decode_attention(qb, Kc, Vc, [4, 4], 2, 1, 1, D, 4, 0.5, var, L=L)
        qh = f16_bits(qb.view(np.float16).astype(np.float64) * 0.5)
        o2 = oracle.decode_attention(qh, Kc, Vc, [4, 4], 2, 1, 1, D, 4, 1.0, var, L=L)
        check(f"attn scale {var}", np.allclose(o1, o2, rtol=1e-15, atol=1e-15))
    # (h) brute force: numpy softmax over dense rows, B = 2, H = 4, Hkv = 2, D = 64
    rng = np.random.default_rng(10)
    for var in (DUAL, FAST):
        B, H, Hkv, D, Tmax = 2, 4, 2, 64, 5
        lens = np.array([5, 3])
        Kc = synth.weights(B * Hkv * Tmax, D, var, seed=6, stream=20)
        Vc = synth.weights(B * Hkv * Tmax, D, var, seed=6, stream=21)
        q = f16_bits(rng.integers(-8, 9, size=(B, H, D)) * 0.125)
        out = oracle.decode_attention(q, Kc, Vc, lens, B, H, Hkv, D, Tmax, 0.125, var, L=L)
        Kd = oracle.dequant(Kc, B * Hkv * Tmax, D, var, L).reshape(B, Hkv, Tmax, D)
        Vd = oracle.dequant(Vc, B * Hkv * Tmax, D, var, L).reshape(B, Hkv, Tmax, D)
        qf = q.view(np.float16).astype(np.float64)
        ok = True
        for b in range(B):
            for h in range(H):
                sc = 0.125 * Kd[b, h // 2, :lens[b]] @ qf[b, h]
                w = np.exp(sc - sc.max())
                ok &= np.allclose(out[b, h], (w @ Vd[b, h // 2, :lens[b]]) / w.sum(), rtol=1e-12, atol=1e-12)
        check(f"attn brute force {var}", ok)


def _pin_quantize(check, L):
    # 11. The quantiser, reading R13 (smallest covering scale, nearest Codebook10
    #     magnitude, ties to the smaller).  Pinned by the decode (pinned above)
    #     and by properties that follow from the rule, not by restating it.
    rng = np.random.default_rng(11)
    for var in (DUAL, FAST):
        bb = synth.block_bytes(var)
        ng = 2 if var == DUAL else 1
        # (a) round trip: blocks whose every scale group holds a code of
        #     magnitude 10 (so the group's scale is the covering one), no code 8
        nblk = 64
        W = np.zeros((nblk, bb), dtype=np.uint8)
        codes = rng.choice(np.r_[0:8, 9:16], size=(nblk, 32))
        for g in range(ng):
            lo = g * (32 // ng)
            codes[:, lo + rng.integers(0, 32 // ng)] = rng.choice([7, 15])
        W[:, :16] = codes[:, :16] | (codes[:, 16:] << 4)
        W[:, 16:] = rng.integers(0x01, 0x7F, size=(nblk, bb - 16))  # finite, nonzero scales
        N, K = 8, nblk // 8 * 32
        Wm = W.reshape(N, -1)
        dense = oracle.dequant(Wm, N, K, var, L)
        # codes up to 10 and half-scales from 2^-10 to 224: every value is exact in fp16
        check(f"quant round trip {var}", np.array_equal(oracle.quantize(f16_bits(dense), N, K, var, L=L), Wm))
        # (b) error bound and minimal scale on random fp16 input
        x = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-12, 10, size=(16, 1)))).astype(np.float16)
        Q = oracle.quantize(x.view(np.uint16), 16, 256, var, L=L)
        back = oracle.dequant(Q, 16, 256, var, L).reshape(16, 8, ng, 32 // ng)
        xs = x.astype(np.float64).reshape(16, 8, ng, 32 // ng)
        sc = Q.reshape(16, 8, bb)[:, :, 16:16 + ng]
        hs = np.vectorize(lambda e: oracle.halfscale(int(e), L))(sc)
        below = np.vectorize(lambda e: oracle.ue4m3(int(e) - 1, L) if e > 0 else 0.0)(sc)
        amax = np.abs(xs).max(axis=3)
        check(f"quant error bound {var}", np.all(np.abs(back - xs) <= hs[..., None] * (1 + 1e-12)))
        check(f"quant minimal scale {var}", np.all((5 * below < amax) | (sc == 0)) and np.all(10 * hs >= amax))
        # (c) sign symmetry: -x flips the sign bit of every nonzero code, same scales
        Qn = oracle.quantize((-x).view(np.uint16), 16, 256, var, L=L).reshape(16, 8, bb)
        Qp = Q.reshape(16, 8, bb)
        lo, hi = Qp[..., :16] & 0xF, Qp[..., :16] >> 4
        flip = lambda c: np.where(c == 0, 0, c ^ 8)
        check(f"quant sign {var}", np.array_equal(Qn[..., 16:], Qp[..., 16:]) and
              np.array_equal(Qn[..., :16] & 0xF, flip(lo)) and np.array_equal(Qn[..., :16] >> 4, flip(hi)))
        # (d) doubling the input adds one to every scale exponent, codes unchanged
        xm = (rng.standard_normal((4, 256)) * 3).astype(np.float16)
        Q1 = oracle.quantize(xm.view(np.uint16), 4, 256, var, L=L).reshape(4, 8, bb)
        Q2 = oracle.quantize((xm * np.float16(2)).view(np.uint16), 4, 256, var, L=L).reshape(4, 8, bb)
        check(f"quant doubling {var}", np.array_equal(Q2[..., :16], Q1[..., :16]) and
              np.array_equal(Q2[..., 16:].astype(int), Q1[..., 16:].astype(int) + 8))
        # (e) the tie rule: with half-scale 1 (group max 10), 5 -> 4, 7 -> 6, 9 -> 8, 0.5 -> 0, 5.5 -> 6
        row = np.zeros(32)
        row[[0, 1, 2, 3, 4, 5]] = [10, 5, 7, 9, 0.5, 5.5]
        if var == DUAL:
            row[16] = 10
        Qt = oracle.quantize(f16_bits(row), 1, 32, var, L=L)[0]
        check(f"quant ties {var}", list(Qt[:6] & 0xF) == [7, 4, 5, 6, 0, 5] and Qt[16] == 0x40)
        # (f) saturation above 5 * 448 = 2240, and zero groups
        row = np.zeros(32)
        row[0], row[1] = 30000.0, -2240.0
        Qs = oracle.quantize(f16_bits(row), 1, 32, var, L=L)[0]
        zero_ok = (Qs[17] == 0 and np.all(Qs[:16] >> 4 == 0)) if var == DUAL else True
        check(f"quant saturation {var}", Qs[16] == 0x7E and Qs[0] & 0xF == 7 and Qs[1] & 0xF == 15 and zero_ok)
