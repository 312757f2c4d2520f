"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix (hand-derived examples, closed forms, invariants, library routines, brute
force on tiny inputs).  CPU only."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oscar_oracle as O
from int2_kv_cache_append_gb300 import synth as S

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))


# --------------------------------------------------------------------------
# number formats against library conversions
# --------------------------------------------------------------------------
def _tricky_f32(n=20000, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n).astype(np.float32) * np.float32(10.0) ** rng.integers(-6, 6, n).astype(np.float32)
    # exact bf16 ties: low 16 bits 0x8000, both parities of the kept lsb
    ties = (rng.integers(0, 2 ** 15, 256).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    return np.concatenate([x, ties, np.array([0.0, -0.0, 1.0, -2.5, 65504.0, 1e-40], np.float32)])


def test_bf16_rounding_matches_torch():
    x = _tricky_f32()
    ours = O.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_fp16_rounding_matches_torch():
    x = _tricky_f32(seed=1)
    x = x[np.abs(x) < 60000]
    ours = x.astype(np.float16).view(np.uint16)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# codec: hand-derived rows
# --------------------------------------------------------------------------
def _row(vals, d=128):
    r = np.zeros((1, d), np.float32)
    r[0, :len(vals)] = vals
    return r


def test_codec_hand_example_ties_to_even():
    # mn=-3, mx=3 -> scale=(3-(-3))/3=2, zero=-3; (x+3)/2: -3->0, -1->1, 1->2, 3->3,
    # 0 -> 1.5 -> 2 (even), -2 -> 0.5 -> 0 (even), 2 -> 2.5 -> 2 (even)
    r = _row([-3, -1, 1, 3, 0, -2, 2])
    codes, sc, ze = O.quantize_rows(r, 1.0)
    assert float(sc[0, 0]) == 2.0 and float(ze[0, 0]) == -3.0
    assert list(codes[0, :7]) == [0, 1, 2, 3, 2, 0, 2]
    assert (codes[0, 7:] == 2).all()  # the zero padding also sits on a tie


def test_codec_clip_bounds_outlier_per_row_not_per_group():
    # D=256: outlier 10 in group 0; group 1 holds values in [-5, 5].
    # Row threshold t = fl32(0.96) * 10 = 9.6 (as float32); group 0's max becomes t,
    # group 1 is untouched because 5 < t.  A per-group clip would shrink group 1.
    d = 256
    r = np.zeros((1, d), np.float32)
    r[0, 0] = 10.0
    r[0, 1] = -1.0
    r[0, 128] = 5.0
    r[0, 129] = -5.0
    codes, sc, ze = O.quantize_rows(r, 0.96)
    t = np.float32(0.96) * np.float32(10.0)
    xh = O.dequantize_rows(codes, sc, ze)
    # group 0: mn=-1, mx=t -> top code reconstructs t up to fp16 rounding of scale/zero
    assert codes[0, 0] == 3
    assert abs(xh[0, 0] - float(t)) <= 3 * abs(float(sc[0, 0]) - (float(t) + 1) / 3) + abs(float(ze[0, 0]) + 1) + 1e-6
    assert abs(xh[0, 0] - 10.0) > 0.3
    # group 1 keeps its full range: zero=-5, scale=10/3 in fp16
    assert float(ze[0, 1]) == -5.0
    assert float(sc[0, 1]) == float(np.float16(np.float32(10.0) / np.float32(3.0)))


def test_codec_constant_group():
    r = np.full((1, 128), 1.5, np.float32)
    codes, sc, ze = O.quantize_rows(r, 1.0)
    assert float(sc[0, 0]) == 0.0 and float(ze[0, 0]) == 1.5 and (codes == 0).all()
    # with a clip ratio the constant row is clipped to ratio*1.5 first
    codes, sc, ze = O.quantize_rows(r, 0.92)
    assert float(ze[0, 0]) == float(np.float16(np.float32(0.92) * np.float32(1.5)))


def test_codec_lattice_rows_round_trip_exactly():
    # x = z + s*c with fp16-exact s and z, extremes present, ratio 1: exact.
    rng = np.random.default_rng(3)
    for _ in range(50):
        d = int(rng.choice([128, 256, 512]))
        rows = []
        for _g in range(d // 128):
            s = float(np.float16(rng.uniform(0.01, 4.0)))
            z = float(np.float16(rng.uniform(-8, 0)))
            c = rng.integers(0, 4, 128)
            c[0], c[1] = 0, 3
            rows.append(z + s * c)
        r = np.concatenate(rows)[None].astype(np.float32)
        # keep the whole row's max |x| as the top value so ratio=1 clips nothing
        codes, sc, ze = O.quantize_rows(r, 1.0)
        xh = O.dequantize_rows(codes, sc, ze)
        assert np.array_equal(xh.astype(np.float32), r), "lattice row not reproduced"


def test_codec_error_bound_and_code_range_random():
    rng = np.random.default_rng(4)
    r = S.activations(rng, (400, 256), [3, 100, 200], kind="t3")
    for ratio in (1.0, 0.96, 0.92):
        codes, sc, ze = O.quantize_rows(r, ratio)
        assert codes.max() <= 3
        a = np.abs(r).max(axis=1)
        t = (np.float32(ratio) * a)[:, None]
        x = np.clip(r, -t, t).astype(np.float64)
        xh = O.dequantize_rows(codes, sc, ze)
        xg = x.reshape(400, 2, 128)
        mn, mx = xg.min(2), xg.max(2)
        s32 = (mx - mn) / 3
        s16 = sc.astype(np.float64)
        z16 = ze.astype(np.float64)
        slack = s16 / 2 + 3 * np.abs(s16 - s32) + np.abs(z16 - mn) + 4 * np.spacing(np.abs(mx).astype(np.float32))
        err = np.abs(xh - x).reshape(400, 2, 128).max(2)
        assert (err <= slack + 1e-7).all()
        # rounding to nearest: most elements sit well inside s/2
        assert np.mean(np.abs(xh - x).reshape(400, 2, 128) <= s16[:, :, None] / 2 + 1e-6) > 0.99


def test_codec_multiplies_by_correctly_rounded_reciprocal():
    # scale 0.88671875 (fp16 0x3B18), zero -0.68408203125 (fp16 0xB979) and the
    # float32 x with bits 0xBE767FFE (found by search): the product with the
    # float32 reciprocal rounds to exactly 0.5, a tie that goes to the even code
    # 0, whereas a true division rounds just above 0.5 and gives code 1.
    s = np.float32(np.uint16(15128).view(np.float16))
    z = np.float32(np.uint16(47481).view(np.float16))
    x = np.array([3195437054], np.uint32).view(np.float32)[0]
    dx = np.float32(x - z)
    via_rcp = np.rint(np.float32(dx * (np.float32(1.0) / s)))
    via_div = np.rint(np.float32(dx / s))
    assert via_rcp == 0.0 and via_div == 1.0          # the two readings disagree here
    # exact rational check of the reciprocal path: 1/s rounded to float32 first,
    # the exact product lies within half a float32 ulp of 1/2, so it rounds to 1/2
    inv = Fraction(float(np.float32(1.0) / s))
    prod = Fraction(float(dx)) * inv
    assert abs(prod - Fraction(1, 2)) <= Fraction(1, 2 ** 26)
    assert Fraction(float(dx)) / Fraction(float(s)) > Fraction(1, 2) + Fraction(1, 2 ** 26)
    row = np.full((1, 128), x, np.float32)
    row[0, 0] = z
    row[0, 1] = np.float32(z + np.float32(3) * s)     # max: scale comes out exactly s
    codes, sc, ze = O.quantize_rows(row, 1.0)
    assert np.float32(sc[0, 0]) == s and np.float32(ze[0, 0]) == z
    assert codes[0, 2] == 0


# --------------------------------------------------------------------------
# physical packing: bytes derived by hand from the documented bit layout
# --------------------------------------------------------------------------
@pytest.mark.parametrize("role,dim,byte,val", [
    (0, 0, 0, 0x01),     # K: dim 0 -> word 0 bit 0
    (0, 1, 2, 0x01),     # K: dim 1 -> word 0 bit 16
    (0, 8, 0, 0x04),     # K: dim 8 = 16*0 + 2*0 + 8*1 -> p=1 -> bit 2
    (0, 2, 8, 0x01),     # K: dim 2 -> c=1 -> word 2 -> byte 8
    (0, 16, 0, 0x10),    # K: dim 16 -> kk=1 -> p=2 -> bit 4
    (0, 64, 4, 0x01),    # K: dim 64 -> kk=4 -> word 1 bit 0
    (0, 15, 14, 0x40),   # K: dim 15 = 14+1 -> c=3,h=1 -> word 6 bit 16+2 -> byte 26? see below
    (1, 0, 0, 0x01),     # V: dim 0 -> word 0 bit 0
    (1, 1, 4, 0x01),     # V: dim 1 -> word 1 (g=1) bit 0
    (1, 8, 0, 0x04),     # V: dim 8 -> g=0, n=1 -> bit 2
    (1, 127, 31, 0x40),  # V: dim 127 = 8*15+7 -> word 7 bit 30 -> byte 31 bit 6
])
def test_pack_layout_hand_bytes(role, dim, byte, val):
    if role == 0 and dim == 15:
        # dim 15 = 16*0 + 2*3 + 8*1 + 1 -> c=3, i=0, p=1 (kk=0,h=1): word 6, bit 16+2=18
        byte, val = 6 * 4 + 2, 0x04
    codes = np.zeros((1, 128), np.uint8)
    codes[0, dim] = 1
    packed = O.pack_codes(codes, role)
    expect = np.zeros(32, np.uint8)
    expect[byte] = val
    assert np.array_equal(packed[0], expect)


def test_pack_second_group_offsets():
    codes = np.zeros((1, 256), np.uint8)
    codes[0, 129] = 3          # V: group 1, g=1, n=0 -> word 9, bits 0-1
    p = O.pack_codes(codes, 1)
    assert p[0, 36] == 3 and p[0].sum() == 3
    p = O.pack_codes(codes, 0)  # K: group 1 dim 1 -> word 8 bit 16 -> byte 34
    assert p[0, 34] == 3 and p[0].sum() == 3


# --------------------------------------------------------------------------
# rotations (generator) and rotation invariance
# --------------------------------------------------------------------------
@pytest.mark.parametrize("d", [128, 256, 512])
def test_hadamard_bitrev_closed_forms(d):
    h = S.hadamard(d)
    assert np.abs(h @ h.T - np.eye(d)).max() < 1e-12
    assert np.all(np.abs(np.abs(h) - 1 / math.sqrt(d)) < 1e-15)
    p = S.bit_reversal(d)
    assert np.array_equal(p @ p, np.eye(d))  # involution


def test_eig_rotation_sorted_eigvecs_and_orthogonal():
    w = S.WORKLOADS["tiny"]
    calib = S.activations(S.rng_for(0, 0, S.ROLE_CALIB), (4096, 128), [3, 17, 90], kind="scale")
    r = S.eig_rotation(calib)
    e = r @ S.bit_reversal(128).T @ S.hadamard(128).T     # undo H P_br
    sig = calib.astype(np.float64).T @ calib.astype(np.float64)
    lam = np.diag(e.T @ sig @ e)
    assert np.all(np.diff(lam) <= 1e-6 * lam[0])
    assert np.abs(sig @ e - e * lam).max() < 1e-6 * lam[0]
    rk, rv = S.rotations(w, 0)
    for R in (rk, rv):
        assert np.abs(R.astype(np.float64) @ R.T.astype(np.float64) - np.eye(128)).max() <= 1e-5


def test_rotation_invariance_of_scores():
    w = S.WORKLOADS["tiny"]
    rk, _ = S.rotations(w, 0)
    rng = np.random.default_rng(5)
    q = rng.standard_normal((8, 128))
    k = rng.standard_normal((64, 128))
    R = rk.astype(np.float64)
    assert np.abs((q @ R) @ (k @ R).T - q @ k.T).max() < 1e-4  # fp32 R: |RR^T - I| ~ 1e-8
    Rx = S.eig_rotation(S.activations(S.rng_for(0, 0, S.ROLE_CALIB), (4096, 128), [3, 17, 90], "scale"))
    assert np.abs((q @ Rx) @ (k @ Rx).T - q @ k.T).max() < 1e-10


# --------------------------------------------------------------------------
# layout against the pages' numbers
# --------------------------------------------------------------------------
def test_layout_compression_matches_pages():
    assert GOLD["group_size"]["value"] == O.GROUP
    d = 128
    int2_row = d // 4 + 4 * (d // O.GROUP)      # codes + fp16 scale + fp16 zero
    ratio = (2 * d) / int2_row
    assert abs(ratio - GOLD["compression_vs_16bit"]["value"]) < 0.25     # "~7x"
    assert (2 * d) / (d // 4) == GOLD["reduction_vs_bf16"]["value"]       # code bits alone: 8x
    layers, hd = GOLD["qwen3_4b_layers_head_dim"]["value"]
    mb = layers * hd * hd * 4 / 1e6                                       # fp32 matrices
    assert abs(mb - GOLD["qwen3_4b_rotation_file_mb"]["value"]) < 0.1
    g = GOLD["gemma_rotation"]["value"]
    assert 512 * 512 * 4 * 18 / 1e6 == pytest.approx(g["size_mb_each"], rel=0.06)  # 48 layers? ~18.9MB


def test_layout_sizes():
    cfg = O.Config(2, 3, 8, 2, 256, 5, 7, 100)
    lay = O.layout(cfg)
    assert lay["ncap"] == 128
    assert lay["sink_bytes"] == O._align(3 * 2 * 5 * 256 * 2)
    assert lay["codes_bytes"] == O._align(3 * 2 * 128 * 64)
    assert lay["sz_bytes"] == O._align(3 * 2 * 128 * 2 * 4)
    assert lay["total_bytes"] == 2 * 2 * lay["role_bytes"]


# --------------------------------------------------------------------------
# append semantics
# --------------------------------------------------------------------------
def _small_cfg(S_=2, W=3, cap=40, D=128, G=2, Hkv=2, B=2):
    return O.Config(1, B, Hkv * G, Hkv, D, S_, W, cap, 0.96, 0.92)


def test_append_ring_slots_hand_example():
    cfg = _small_cfg(S_=2, W=3, B=1, Hkv=1, G=1)
    cache = O.new_cache(cfg)
    I = np.eye(128, dtype=np.float32)
    for p in range(7):
        k = np.full((1, 1, 1, 128), p + 1.0, np.float32)
        O.append(cfg, cache, 0, k, k, [p], I, I)
    v = O.CacheView(cfg, cache, 0, 0)
    got = O.bf16_bits_to_f32(v.ring[0, 0, :, 0])
    assert list(got) == [7.0, 5.0, 6.0]      # slots 0,1,2 <- tokens 6,4,5 (values p+1)
    assert list(O.bf16_bits_to_f32(v.sink[0, 0, :, 0])) == [1.0, 2.0]


def test_append_skips_positions_beyond_capacity():
    # capacity 5, S=2, W=2: tokens at positions 3..7 -> only 3 and 4 are stored
    cfg = _small_cfg(S_=2, W=2, cap=5, B=1, Hkv=1, G=1)
    cache = O.new_cache(cfg)
    I = np.eye(128, dtype=np.float32)
    k = (np.arange(5, dtype=np.float32) + 10.0)[None, :, None, None] * np.ones((1, 5, 1, 128), np.float32)
    O.append(cfg, cache, 0, k, k, [3], I, I)
    v = O.CacheView(cfg, cache, 0, 0)
    assert O.layout(cfg)["ncap"] == 64      # rows exist past capacity in memory ...
    zq = v.sz[0, 0, :, 0, 1].astype(np.float64)
    assert zq[1] != 0 and zq[2] != 0       # positions 3, 4 (rows 1, 2) written
    assert np.all(zq[3:] == 0)             # ... but positions 5.. are never written
    # ring slots hold the last W=2 stored tokens only if they are in the cache:
    # newlen - W = 6 -> positions 6, 7 are beyond capacity, so the ring stays empty
    assert np.all(v.ring == 0)


def test_append_chunking_invariance():
    cfg = _small_cfg(S_=3, W=5, cap=64)
    rng = np.random.default_rng(6)
    rk = S.qr_rotation(rng, 128).astype(np.float32)
    rv = S.qr_rotation(rng, 128).astype(np.float32)
    T = 29
    k = S.to_bf16_values(rng.standard_normal((2, T, 2, 128)).astype(np.float32))
    v = S.to_bf16_values(rng.standard_normal((2, T, 2, 128)).astype(np.float32))
    c1 = O.new_cache(cfg)
    O.append(cfg, c1, 0, k, v, [0, 0], rk, rv)
    c2 = O.new_cache(cfg)
    pos = 0
    for n in (1, 4, 2, 7, 1, 14):
        O.append(cfg, c2, 0, k[:, pos:pos + n], v[:, pos:pos + n], [pos, pos], rk, rv)
        pos += n
    assert pos == T
    q = S.to_bf16_values(rng.standard_normal((2, 4, 128)).astype(np.float32))
    o1, l1 = O.decode(cfg, c1, 0, q, [T, T], rk, rv)
    o2, l2 = O.decode(cfg, c2, 0, q, [T, T], rk, rv)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# --------------------------------------------------------------------------
# attention: library routine, closed forms, brute force
# --------------------------------------------------------------------------
def test_all_bf16_window_equals_library_sdpa():
    # S + W >= T: every token is BF16; with R = I the result is plain scaled
    # dot-product attention over BF16(K), BF16(V) (torch reference, float64).
    cfg = _small_cfg(S_=8, W=16, cap=64, G=3, Hkv=2, B=2)
    rng = np.random.default_rng(7)
    T = 20
    k = S.to_bf16_values(rng.standard_normal((2, T, 2, 128)).astype(np.float32) * 2)
    v = S.to_bf16_values(rng.standard_normal((2, T, 2, 128)).astype(np.float32))
    I = np.eye(128, dtype=np.float32)
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k, v, [0, 0], I, I)
    q = S.to_bf16_values(rng.standard_normal((2, 6, 128)).astype(np.float32))
    out, lse = O.decode(cfg, cache, 0, q, [T, T], I, I)
    qt = torch.from_numpy(q.astype(np.float64))[:, :, None, :]             # B,Hq,1,D
    kt = torch.from_numpy(k.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(3, dim=1)
    vt = torch.from_numpy(v.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(3, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, :, 0].numpy()
    assert np.abs(out - ref).max() < 1e-12
    sc = torch.einsum("bhd,bhtd->bht", qt[:, :, 0], kt) / math.sqrt(128)
    assert np.abs(lse - torch.logsumexp(sc, dim=-1).numpy()).max() < 1e-12


def _signed_permutation(rng, d):
    # a random permutation matrix with random signs (orthogonal, not symmetric):
    # every product with it is exact in every float format
    P = np.zeros((d, d), np.float32)
    P[np.arange(d), rng.permutation(d)] = rng.choice([-1.0, 1.0], d)
    assert not np.array_equal(P, P.T)
    return P


def _symmetric_lattice_rotated_rows(rng, shape):
    # rows in the rotated basis: per 128-group values in {-3s/2, -s/2, s/2, 3s/2}
    # (s a power of two, both extremes present): exact in bf16 and fp16, and the
    # codec (clip ratio 1) returns them exactly (scale s, zero -3s/2, codes 0..3)
    x = np.empty(shape, dtype=np.float32)
    D = shape[-1]
    for idx in np.ndindex(*shape[:-1]):
        for j in range(D // 128):
            s = float(rng.choice([0.25, 0.5, 1.0, 2.0]))
            c = rng.integers(0, 4, 128)
            c[0], c[1] = 0, 3
            x[idx][128 * j:128 * (j + 1)] = s * (c - 1.5)
    return x


@pytest.mark.parametrize("D", [128, 256])
def test_rotated_cache_decode_equals_sdpa_on_unrotated_rows(D):
    # Gemma card [Folders]: the rotation applies to Q/K (and V); so q'.k' = q.k and
    # the output is un-rotated.  With signed-permutation R_K, R_V (exact) and rows
    # whose rotated images are exact in every storage form (BF16 windows and the
    # INT2 region alike, clip ratio 1), append + decode through the rotations must
    # equal plain attention over the UNROTATED K and V.
    B, H, G, T = 2, 2, 2, 40
    cfg = O.Config(1, B, H * G, H, D, 4, 6, 64, 1.0, 1.0)
    rng = np.random.default_rng(71 + D)
    RK, RV = _signed_permutation(rng, D), _signed_permutation(rng, D)
    rk = _symmetric_lattice_rotated_rows(rng, (B, T, H, D))
    rv = _symmetric_lattice_rotated_rows(rng, (B, T, H, D))
    k = (rk.astype(np.float64) @ RK.T.astype(np.float64)).astype(np.float32)  # k R_K = rk exactly
    v = (rv.astype(np.float64) @ RV.T.astype(np.float64)).astype(np.float32)
    q = S.to_bf16_values(rng.standard_normal((B, H * G, D)).astype(np.float32))
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k, v, [0, 0], RK, RV)
    lens = [T, 23]
    for absorb in (False, True):
        out, lse = O.decode(cfg, cache, 0, q, lens, RK, RV, absorb_v=absorb)
        for b in range(B):
            Tb = lens[b]
            if b == 1:  # the ring holds the last W appended positions: only T is fully windowed
                continue
            qt = torch.from_numpy(q[b].astype(np.float64))[:, None, :]
            kt = torch.from_numpy(k[b, :Tb].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
            vt = torch.from_numpy(v[b, :Tb].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0].numpy()
            if absorb:  # the rotated basis: o' = o R_V
                ref = ref @ RV.astype(np.float64)
            assert np.abs(out[b] - ref).max() < 1e-12 * max(1.0, np.abs(ref).max())
            sc = torch.einsum("hd,htd->ht", qt[:, 0], kt) / math.sqrt(D)
            assert np.abs(lse[b] - torch.logsumexp(sc, -1).numpy()).max() < 1e-12


def test_qr_rotated_bf16_windows_equal_sdpa_on_unrotated_rows_within_bf16_rounding():
    # S + W >= T, calibrated-like (QR) rotations: the cache holds BF16(k R_K) and
    # BF16(v R_V); decode must equal attention over the unrotated K and V up to
    # the BF16 rounding of the rotated rows.  Bound, with u = 2^-9 (BF16 unit
    # roundoff) and eps = max_t |score perturbation| <= sm_scale |q| u |k_t|:
    #   |out - ref| <= (e^{2 eps} - 1) (max_t |v_t - c| + u max_t |v_t|_2) + u max_t |v_t|_2,
    #   |lse - ref| <= eps,
    # c any per-channel constant (the weight changes sum to zero): the midrange
    B, H, G, D, T = 2, 2, 3, 128, 30
    cfg = O.Config(1, B, H * G, H, D, 10, 24, 64, 0.96, 0.92)
    rng = np.random.default_rng(77)
    RK, RV = S.qr_rotation(rng, D).astype(np.float32), S.qr_rotation(rng, D).astype(np.float32)
    k = S.to_bf16_values(rng.standard_normal((B, T, H, D)).astype(np.float32))
    # V rows with a common offset: a wrong un-rotation moves the output by about the offset
    v = S.to_bf16_values(rng.standard_normal((B, T, H, D)).astype(np.float32) + np.float32(2.0))
    q = S.to_bf16_values(rng.standard_normal((B, H * G, D)).astype(np.float32) * np.float32(0.5))
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k, v, [0, 0], RK, RV)
    out, lse = O.decode(cfg, cache, 0, q, [T, T], RK, RV)
    u = 2.0 ** -9 * (1 + 2.0 ** -14)  # BF16 rounding, plus the float32 rounding of the rotated row
    for b in range(B):
        qt = torch.from_numpy(q[b].astype(np.float64))[:, None, :]
        kt = torch.from_numpy(k[b].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        vt = torch.from_numpy(v[b].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0].numpy()
        sc = torch.einsum("hd,htd->ht", qt[:, 0], kt) / math.sqrt(D)
        qn = np.linalg.norm(q[b].astype(np.float64), axis=1)                      # [Hq]
        kn = np.linalg.norm(k[b].astype(np.float64), axis=2)                      # [T, H]
        vn = np.linalg.norm(v[b].astype(np.float64), axis=2)
        for i in range(H * G):
            h = i // G
            eps = qn[i] * u * kn[:, h].max() / math.sqrt(D)
            vh = v[b, :, h].astype(np.float64)
            c = (vh.max(0) + vh.min(0)) / 2
            bound = (math.exp(2 * eps) - 1) * (np.abs(vh - c).max() + u * vn[:, h].max()) + u * vn[:, h].max()
            err = np.abs(out[b, i] - ref[i]).max()
            assert err <= bound, (b, i, err, bound)
            assert abs(lse[b, i] - float(torch.logsumexp(sc[i], -1))) <= eps
        # the bound is small against the output (a transposed rotation moves it by ~2)
        assert bound < 0.25 * np.abs(ref).min()


def test_uniform_attention_window_boundaries_closed_form():
    # K = 0 -> uniform attention; V rows constant p+1 per token.  BF16 tokens keep
    # p+1; INT2 tokens hold the constant-row codec value fp16(fl32(ratio*(p+1))).
    for (S_, W, T) in [(4, 6, 30), (0, 5, 17), (3, 0, 12), (5, 5, 9), (8, 4, 6), (2, 3, 3)]:
        cfg = _small_cfg(S_=S_, W=W, cap=64, G=1, Hkv=1, B=1)
        I = np.eye(128, dtype=np.float32)
        cache = O.new_cache(cfg)
        k = np.zeros((1, T, 1, 128), np.float32)
        v = np.broadcast_to((np.arange(T, dtype=np.float32) + 1)[None, :, None, None], (1, T, 1, 128)).copy()
        O.append(cfg, cache, 0, k, v, [0], I, I)
        q = np.ones((1, 1, 128), np.float32)
        out, lse = O.decode(cfg, cache, 0, q, [T], I, I)
        total = 0.0
        for p in range(T):
            in_sink = p < S_
            in_ring = p >= max(S_, T - W)
            if in_sink or in_ring:
                total += p + 1
            else:
                total += float(np.float16(np.float32(0.92) * np.float32(p + 1)))
        assert abs(out[0, 0, 0] - total / T) < 1e-12, (S_, W, T)
        assert abs(lse[0, 0] - math.log(T)) < 1e-12


def test_one_hot_and_constant_v():
    cfg = _small_cfg(S_=2, W=2, cap=64, G=2, Hkv=1, B=1)
    rng = np.random.default_rng(8)
    T = 40
    I = np.eye(128, dtype=np.float32)
    k = S.to_bf16_values(rng.standard_normal((1, T, 1, 128)).astype(np.float32))
    k[0, 17, 0, :] = 0
    k[0, 17, 0, 5] = 200.0      # one token with a huge logit (INT2 region)
    vrow = np.float32(0.5) * np.arange(128, dtype=np.float32) % np.float32(4.0) - np.float32(1.0)
    v = np.broadcast_to(vrow, (1, T, 1, 128)).copy()
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k, v, [0], I, I)
    q = np.zeros((1, 2, 128), np.float32)
    q[0, 0, 5] = 50.0
    out, _ = O.decode(cfg, cache, 0, q, [T], I, I)
    # head 0: all weight on token 17 -> its INT2 reconstruction of vrow
    expect17 = O.dequant_history(cfg, cache, 0, 1, 0, 0, T)[17]
    assert np.abs(out[0, 0] - expect17).max() < 1e-9
    # head 1 (q=0): uniform average; the constant V row: BF16 tokens give vrow,
    # INT2 tokens give the same reconstruction each -> a closed-form mean
    nb = 2 + 2
    expect = (nb * vrow.astype(np.float64) + (T - nb) * expect17) / T
    assert np.abs(out[0, 1] - expect).max() < 1e-12


def test_decode_brute_force_tiny():
    # Pure-Python loops, independent of the oracle's vectorised path.
    cfg = _small_cfg(S_=2, W=3, cap=64, G=2, Hkv=2, B=2)
    rng = np.random.default_rng(9)
    T = [11, 7]
    rk = S.qr_rotation(rng, 128).astype(np.float32)
    rv = S.qr_rotation(rng, 128).astype(np.float32)
    k = S.to_bf16_values(rng.standard_normal((2, 11, 2, 128)).astype(np.float32))
    v = S.to_bf16_values(rng.standard_normal((2, 11, 2, 128)).astype(np.float32))
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k[:, :7], v[:, :7], [0, 0], rk, rv)
    # both rows get 4 more tokens; row b=1 is then decoded with T=7, which must
    # ignore every position >= 7
    c2 = cache.copy()
    O.append(cfg, c2, 0, k[:, 7:], v[:, 7:], [7, 7], rk, rv)
    # row b=1 must look as if it had 7 tokens: decode with T=7 ignores positions >= 7
    q = S.to_bf16_values(rng.standard_normal((2, 4, 128)).astype(np.float32))
    out, lse = O.decode(cfg, c2, 0, q, T, rk, rv, absorb_v=False)
    for b in range(2):
        for i in range(4):
            h = i // 2
            K = O.dequant_history(cfg, c2, 0, 0, b, h, T[b])
            V = O.dequant_history(cfg, c2, 0, 1, b, h, T[b])
            qr = [sum(float(q[b, i, a]) * float(rk[a, j]) for a in range(128)) for j in range(128)]
            sc = [sum(qr[j] * K[t, j] for j in range(128)) / math.sqrt(128) for t in range(T[b])]
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            l = sum(e)
            orot = [sum(e[t] * V[t, j] for t in range(T[b])) / l for j in range(128)]
            o = [sum(orot[j] * float(rv[a, j]) for j in range(128)) for a in range(128)]
            assert max(abs(o[a] - out[b, i, a]) for a in range(128)) < 1e-11
            assert abs(m + math.log(l) - lse[b, i]) < 1e-11


def test_absorb_v_is_output_in_rotated_basis():
    cfg = _small_cfg(S_=2, W=3, cap=64)
    rng = np.random.default_rng(10)
    rk = S.qr_rotation(rng, 128).astype(np.float32)
    rv = S.qr_rotation(rng, 128).astype(np.float32)
    k = S.to_bf16_values(rng.standard_normal((2, 20, 2, 128)).astype(np.float32))
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k, k[:, ::-1].copy(), [0, 0], rk, rv)
    q = S.to_bf16_values(rng.standard_normal((2, 4, 128)).astype(np.float32))
    o_abs, l1 = O.decode(cfg, cache, 0, q, [20, 13], rk, rv, absorb_v=True)
    o, l2 = O.decode(cfg, cache, 0, q, [20, 13], rk, rv, absorb_v=False)
    assert np.abs(o_abs @ rv.astype(np.float64).T - o).max() < 1e-12
    assert np.array_equal(l1, l2)


# --------------------------------------------------------------------------
# data-free in-quant Hadamard (FLAG_HADAMARD)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("d", [128, 256, 512])
def test_in_quant_hadamard_is_block_diagonal_sylvester(d):
    # each 128-channel block is scipy's Sylvester-ordered Hadamard matrix / sqrt(128);
    # everything off the diagonal blocks is zero; the whole matrix is orthogonal
    L = pytest.importorskip("scipy.linalg")
    H = O.hadamard_rotation(d)
    ref = L.hadamard(128).astype(np.float64) / math.sqrt(128)
    for a in range(d // 128):
        for b in range(d // 128):
            blk = H[128 * a:128 * (a + 1), 128 * b:128 * (b + 1)]
            assert np.array_equal(blk, ref if a == b else np.zeros((128, 128)))
    assert np.abs(H @ H.T - np.eye(d)).max() < 1e-12
    assert np.array_equal(H, H.T)


def test_in_quant_hadamard_hand_entries():
    # Walsh rows by hand: row 0 all +, row 1 alternates, row 2 in pairs, row 3 = row1*row2
    H = O.hadamard_rotation(128) * math.sqrt(128)
    assert np.all(H[0] == 1)
    assert list(H[1, :4]) == [1, -1, 1, -1]
    assert list(H[2, :4]) == [1, 1, -1, -1]
    assert list(H[3, :4]) == [1, -1, -1, 1]
    assert H[127, 127] == -1 and H[64, 63] == 1 and H[64, 64] == -1


def test_hadamard_flag_ignores_given_rotations():
    # the flag rotates by the Hadamard whatever R_K / R_V say: same bytes and
    # outputs as passing the Hadamard explicitly without the flag
    cfg = _small_cfg(S_=4, W=8, cap=64, G=2, Hkv=2, B=2)
    cfg_h = _small_cfg(S_=4, W=8, cap=64, G=2, Hkv=2, B=2)
    cfg_h.flags = O.FLAG_HADAMARD
    rng = np.random.default_rng(21)
    k = S.to_bf16_values(rng.standard_normal((2, 30, 2, 128)).astype(np.float32))
    v = S.to_bf16_values(rng.standard_normal((2, 30, 2, 128)).astype(np.float32))
    q = S.to_bf16_values(rng.standard_normal((2, 4, 128)).astype(np.float32))
    H = O.hadamard_rotation(128)
    junk = rng.standard_normal((128, 128)).astype(np.float32)
    c1, c2 = O.new_cache(cfg), O.new_cache(cfg_h)
    O.append(cfg, c1, 0, k, v, [0, 0], H, H)
    O.append(cfg_h, c2, 0, k, v, [0, 0], junk, None)
    assert np.array_equal(c1, c2)
    o1, l1 = O.decode(cfg, c1, 0, q, [30, 17], H, H)
    o2, l2 = O.decode(cfg_h, c2, 0, q, [30, 17], None, junk)
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l1 - l2).max() < 1e-12


@pytest.mark.parametrize("j", [0, 1, 77])
def test_hadamard_spreads_a_one_hot_row_to_two_levels(j):
    # a one-hot row c e_j becomes c H[j] = +-c/sqrt(128) on every channel: after
    # the 0.96 clip it has two levels, so every code is 0 or 3 (Walsh rows j > 0
    # have 64 of each sign); row 0 is constant, so its group has scale 0, codes 0
    cfg = _small_cfg(S_=0, W=0, cap=64, G=1, Hkv=1, B=1)
    cfg.flags = O.FLAG_HADAMARD
    x = np.zeros((1, 1, 1, 128), dtype=np.float32)
    x[..., j] = 4.0
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, x, x, [0], None, None)
    for role in (0, 1):
        view = O.CacheView(cfg, cache, 0, role)
        codes = O.unpack_codes(view.codes[0, 0, :1], 128, role)[0]
        scale, zero = float(view.sz[0, 0, 0, 0, 0]), float(view.sz[0, 0, 0, 0, 1])
        t = np.float32(0.96 if role == 0 else cfg.v_clip) * np.float32(4.0 / math.sqrt(128))
        if j == 0:
            assert np.all(codes == 0) and scale == 0.0 and zero == float(np.float16(t))
        else:
            assert set(np.unique(codes)) == {0, 3} and int((codes == 3).sum()) == 64
            signs = O.hadamard_rotation(128)[j] > 0
            assert np.array_equal(codes == 3, signs)
            assert zero == float(np.float16(-t))


# --------------------------------------------------------------------------
# K-only INT2 (FLAG_V_BF16): V kept BF16 at every position
# --------------------------------------------------------------------------
def test_v_bf16_layout_sizes():
    base = O.Config(3, 2, 8, 4, 256, 16, 32, 1000, 0.96, 0.92)
    vb = O.Config(3, 2, 8, 4, 256, 16, 32, 1000, 0.96, 0.92, flags=O.FLAG_V_BF16)
    a, b = O.layout(base), O.layout(vb)
    for key in ("ncap", "sink_bytes", "ring_bytes", "codes_bytes", "sz_bytes", "role_bytes"):
        assert a[key] == b[key]                                   # the K role is unchanged
    v = 2 * 4 * 1000 * 256 * 2                                    # one bf16 row per position
    assert b["v_role_bytes"] == -(-v // 256) * 256
    assert b["layer_bytes"] == b["role_bytes"] + b["v_role_bytes"]
    assert b["total_bytes"] == 3 * b["layer_bytes"]
    assert a["v_role_bytes"] == a["role_bytes"] and a["layer_bytes"] == 2 * a["role_bytes"]


def _exact_lattice_rows(rng, shape):
    # per 128-group x = z + s c with s, z and every x exact in fp16 and bf16 and
    # codes 0 and 3 present: the codec (clip ratio 1) and the BF16 windows both
    # return x exactly
    B, T, H, D = shape
    x = np.empty(shape, dtype=np.float32)
    for idx in np.ndindex(B, T, H):
        for j in range(D // 128):
            s = float(rng.choice([0.25, 0.5, 0.75, 1.25]))
            z = float(rng.choice([-3.0, -2.0, -1.5, -0.75]))
            c = rng.integers(0, 4, 128)
            c[0], c[1] = 0, 3
            x[idx][128 * j:128 * (j + 1)] = z + s * c
    return x


def test_v_bf16_decode_equals_library_sdpa_on_exact_k():
    # with K exact in every storage form and V kept BF16, the decode over every
    # position (sink, INT2 region and ring alike) is plain attention over (K, V)
    B, H, G, D, T = 2, 2, 2, 128, 40
    cfg = O.Config(1, B, H * G, H, D, 4, 6, 64, 1.0, 0.92, flags=O.FLAG_V_BF16)
    rng = np.random.default_rng(31)
    k = _exact_lattice_rows(rng, (B, T, H, D))
    v = S.to_bf16_values(rng.standard_normal((B, T, H, D)).astype(np.float32))
    q = S.to_bf16_values(rng.standard_normal((B, H * G, D)).astype(np.float32))
    I = np.eye(D, dtype=np.float32)
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k, v, [0, 0], I, I)
    lens = [T, T]  # the ring holds the last W appended positions: decode at the appended length
    out, lse = O.decode(cfg, cache, 0, q, lens, I, I)
    for b in range(B):
        Tb = lens[b]
        qt = torch.from_numpy(q[b].astype(np.float64))[:, None, :]                       # Hq,1,D
        kt = torch.from_numpy(k[b, :Tb].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        vt = torch.from_numpy(v[b, :Tb].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0].numpy()
        assert np.abs(out[b] - ref).max() < 1e-12
        sc = torch.einsum("hd,htd->ht", qt[:, 0], kt) / math.sqrt(D)
        assert np.abs(lse[b] - torch.logsumexp(sc, -1).numpy()).max() < 1e-12


def test_v_bf16_equals_int2_v_mode_when_everything_is_in_the_windows():
    # S + W >= T: both modes attend BF16 copies of the same rotated rows
    rng = np.random.default_rng(32)
    k = S.to_bf16_values(rng.standard_normal((2, 30, 2, 128)).astype(np.float32))
    v = S.to_bf16_values(rng.standard_normal((2, 30, 2, 128)).astype(np.float32))
    q = S.to_bf16_values(rng.standard_normal((2, 4, 128)).astype(np.float32))
    rk, rv = S.qr_rotation(rng, 128).astype(np.float32), S.qr_rotation(rng, 128).astype(np.float32)
    outs = []
    for flags in (0, O.FLAG_V_BF16):
        cfg = O.Config(1, 2, 4, 2, 128, 10, 20, 64, 0.96, 0.92, flags=flags)
        cache = O.new_cache(cfg)
        O.append(cfg, cache, 0, k, v, [0, 0], rk, rv)
        outs.append(O.decode(cfg, cache, 0, q, [30, 17], rk, rv))
    assert np.abs(outs[0][0] - outs[1][0]).max() < 1e-12
    assert np.abs(outs[0][1] - outs[1][1]).max() < 1e-12


# --------------------------------------------------------------------------
# calibration of R_K (NEXT row f4)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [2, 8, 128, 512])
def test_sylvester_hadamard_matches_scipy(n):
    L = pytest.importorskip("scipy.linalg")
    assert np.abs(O.sylvester_hadamard(n) - L.hadamard(n) / math.sqrt(n)).max() < 1e-15


@pytest.mark.parametrize("d", [128, 256])
def test_calibrate_rk_diagonal_closed_form(d):
    # rows that are scaled unit vectors give a diagonal Sigma with distinct
    # entries: E is the permutation sorting the channels by scale, so
    # R[i][j] = (-1)^popcount(rank(i) & br(j)) / sqrt(d), written out by hand
    rng = np.random.default_rng(41)
    scale = rng.permutation(np.arange(1, d + 1)).astype(np.float64)
    q = np.zeros((2 * d, d))
    for i in range(d):
        q[2 * i, i] = scale[i]
        q[2 * i + 1, i] = -scale[i]
    R = O.calibrate_rk(q)
    order = sorted(range(d), key=lambda i: -scale[i])
    rank = {ch: r for r, ch in enumerate(order)}
    bits = d.bit_length() - 1
    br = [int(format(j, f"0{bits}b")[::-1], 2) for j in range(d)]
    for i in range(d):
        for j in range(0, d, 7):
            want = (-1.0) ** bin(rank[i] & br[j]).count("1") / math.sqrt(d)
            assert abs(R[i, j] - want) < 1e-12


def test_calibrate_rk_eigen_equation_order_and_signs():
    # undo H P_br (scipy's Hadamard): the columns of E must satisfy Sigma e = lambda e,
    # with lambda descending and each column's largest |entry| positive
    L = pytest.importorskip("scipy.linalg")
    d = 128
    calib = S.activations(np.random.default_rng(42), (3000, d), [5, 40, 99], kind="t3")
    R = O.calibrate_rk(calib)
    bits = d.bit_length() - 1
    P = np.zeros((d, d))
    for i in range(d):
        P[i, int(format(i, f"0{bits}b")[::-1], 2)] = 1.0
    E = R @ P.T @ (L.hadamard(d) / math.sqrt(d)).T
    sig = calib.astype(np.float64).T @ calib.astype(np.float64)
    lam = np.einsum("ij,ij->j", E, sig @ E)
    assert np.abs(sig @ E - E * lam).max() < 1e-9 * lam[0]
    assert np.all(np.diff(lam) <= 1e-9 * lam[0])
    assert np.abs(E.T @ E - np.eye(d)).max() < 1e-12
    piv = np.argmax(np.abs(E), axis=0)
    assert np.all(E[piv, np.arange(d)] > 0)


# --------------------------------------------------------------------------
# Lloyd-Max levels (FLAG_LLOYD_MAX)
# --------------------------------------------------------------------------
def test_lloyd_max_ratio_is_the_gaussian_lloyd_max_gap_ratio():
    # Lloyd's iteration for four levels of N(0, 1) (centroid of each cell from the
    # normal density, boundaries at the midpoints) converges to +-0.4528, +-1.5104;
    # its outer gap over its inner gap is the ratio the pages set to 1.16, and the
    # oracle's levels have gaps (rho, 1, rho) with rho that value
    norm = pytest.importorskip("scipy.stats").norm
    lv = np.array([-2.0, -0.5, 0.5, 2.0])
    for _ in range(500):
        b = np.concatenate([[-np.inf], (lv[:-1] + lv[1:]) / 2, [np.inf]])
        lv = (norm.pdf(b[:-1]) - norm.pdf(b[1:])) / (norm.cdf(b[1:]) - norm.cdf(b[:-1]))
    assert abs(lv[3] - 1.5104) < 1e-3 and abs(lv[2] - 0.4528) < 1e-3
    gauss_ratio = (lv[3] - lv[2]) / (lv[2] - lv[1])
    lev = O.lloyd_max_levels()
    gaps = np.diff(lev)
    assert lev[0] == 0.0 and gaps[1] == 1.0 and gaps[0] == gaps[2] == O.LM_RATIO
    # the ratio is the printed one, rounded once to float32
    assert O.LM_RATIO == float(np.float32(GOLD["lm_ratio"]["value"]))
    assert abs(O.LM_RATIO - gauss_ratio) < 0.01
    # span and midpoints: float32 roundings of the exact values of the levels
    # (the span and the first two midpoints are exact, the third one rounding)
    span, mids = O.lloyd_max_thresholds()
    rho = Fraction(O.LM_RATIO)
    assert Fraction(float(span)) == 2 * rho + 1
    exact_mids = [rho / 2, rho + Fraction(1, 2), 3 * rho / 2 + 1]
    assert Fraction(float(mids[0])) == exact_mids[0] and Fraction(float(mids[1])) == exact_mids[1]
    assert float(mids[2]) == float(np.float32(float(exact_mids[2])))
    ulp = Fraction(float(np.spacing(np.float32(mids[2]))))
    assert abs(Fraction(float(mids[2])) - exact_mids[2]) <= ulp / 2


def test_lloyd_max_codec_hand_example():
    # group 0 spans 0 .. 2 rho + 1 (exact in float32), so the unit is exactly 1 and
    # the zero 0 and y = x: the float32 level midpoints rho/2, rho + 1/2 and
    # RN(3 rho/2 + 1) split the codes; a value on a midpoint takes the lower
    # level, its float32 neighbours fall either side
    rho32 = np.float32(O.LM_RATIO)
    rho = Fraction(O.LM_RATIO)
    span = float(np.float32(2) * rho32 + np.float32(1))
    assert Fraction(span) == 2 * rho + 1
    up = lambda v: float(np.nextafter(np.float32(v), np.float32(10)))
    dn = lambda v: float(np.nextafter(np.float32(v), np.float32(-10)))
    m1 = float(rho32 * np.float32(0.5))
    m2 = float(rho32 + np.float32(0.5))
    m3 = float(np.float32(span) - np.float32(m1))
    lev2 = float(np.float32(float(rho + 1)))  # rho + 1 needs 25 bits: its float32 neighbour
    vals = [0.0, span,
            dn(m1), m1, up(m1),
            float(rho32), dn(m2), m2, up(m2),
            lev2, dn(m3), m3, up(m3)]
    r = _row(vals)
    codes, sc, ze = O.quantize_rows(r, 1.0, lloyd_max=True)
    assert float(sc[0, 0]) == 1.0 and float(ze[0, 0]) == 0.0
    assert list(codes[0, :13]) == [0, 3, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2, 3]
    assert (codes[0, 13:] == 0).all()
    xh = O.dequantize_rows(codes, sc, ze, lloyd_max=True)
    assert [Fraction(v) for v in xh[0, [0, 5, 9, 1]]] == [0, rho, rho + 1, 2 * rho + 1]


def _lm_lattice_rows(rng, shape):
    # per 128-group x = u * (level(c) - k) with u = 2^e (e in -6..2) and k in 1..3,
    # codes 0 and 3 present: level - k is rho - k, rho + 1 - k, 2 rho + 1 - k or
    # -k, each exact in float32 (24 significant bits of rho, shifted), and so is the
    # span u (2 rho + 1); the unit u and zero -u k are exact in fp16, so the codec
    # (clip ratio 1) returns x exactly although x - zero = u (rho + 1) is not
    lev = O.lloyd_max_levels()
    x = np.empty(shape, dtype=np.float32)
    D = shape[-1]
    for idx in np.ndindex(*shape[:-1]):
        for j in range(D // 128):
            u = 2.0 ** int(rng.integers(-6, 3))
            kz = int(rng.integers(1, 4))
            c = rng.integers(0, 4, 128)
            c[0], c[1] = 0, 3
            vals = u * (lev[c] - kz)
            assert np.array_equal(vals.astype(np.float32).astype(np.float64), vals)
            x[idx][128 * j:128 * (j + 1)] = vals
    return x


def test_lloyd_max_lattice_rows_round_trip_exactly():
    rng = np.random.default_rng(13)
    for d in (128, 256, 512):
        r = _lm_lattice_rows(rng, (40, d))
        codes, sc, ze = O.quantize_rows(r, 1.0, lloyd_max=True)
        xh = O.dequantize_rows(codes, sc, ze, lloyd_max=True)
        assert np.array_equal(xh, r.astype(np.float64))
        # the uniform codec does not reproduce these rows
        cu, su, zu = O.quantize_rows(r, 1.0)
        assert not np.array_equal(O.dequantize_rows(cu, su, zu), r.astype(np.float64))


def test_lloyd_max_codes_are_nearest_levels_and_error_bound():
    rng = np.random.default_rng(14)
    n, d = 300, 256
    r = S.activations(rng, (n, d), [3, 100, 200], kind="t3")
    lev = O.lloyd_max_levels()
    rho = O.LM_RATIO
    for ratio in (1.0, 0.96, 0.92):
        codes, sc, ze = O.quantize_rows(r, ratio, lloyd_max=True)
        t = (np.float32(ratio) * np.abs(r).max(axis=1))[:, None]
        x = np.clip(r, -t, t).astype(np.float64).reshape(n, 2, 128)
        u = sc.astype(np.float64)[:, :, None]
        z = ze.astype(np.float64)[:, :, None]
        # brute force: distance to each of the four levels, in float64
        dist = np.abs(x[..., None] - (z[..., None] + u[..., None] * lev))
        best = dist.min(-1)
        mine = np.take_along_axis(dist, codes.reshape(n, 2, 128)[..., None].astype(np.int64), -1)[..., 0]
        # the codec decides in float32: a different choice only within rounding of a tie
        assert np.all(mine - best <= 1e-5 * u)
        assert np.mean(mine == best) > 0.999
        # error bound: half the outer gap plus the fp16 rounding of unit and zero
        mn, mx = x.min(2), x.max(2)
        s32 = (mx - mn) / (2 * rho + 1)
        slack = (sc.astype(np.float64) * rho / 2 + (2 * rho + 1) * np.abs(sc.astype(np.float64) - s32)
                 + np.abs(ze.astype(np.float64) - mn) + 1e-6 * np.abs(mx))
        xh = O.dequantize_rows(codes, sc, ze, lloyd_max=True).reshape(n, 2, 128)
        assert (np.abs(xh - x).max(2) <= slack).all()


def test_lloyd_max_lowers_squared_error_on_gaussian_rows():
    # levels shaped like the Gaussian Lloyd-Max quantiser fit Gaussian rows better
    # than evenly spaced ones over the same min..max; the inverse shape (wide
    # middle gap) does worse, so this fixes which gap rho multiplies
    rng = np.random.default_rng(15)
    r = rng.standard_normal((2000, 128)).astype(np.float32)
    cu, su, zu = O.quantize_rows(r, 1.0)
    cl, sl, zl = O.quantize_rows(r, 1.0, lloyd_max=True)
    mse_u = np.mean((O.dequantize_rows(cu, su, zu) - r) ** 2)
    mse_l = np.mean((O.dequantize_rows(cl, sl, zl, lloyd_max=True) - r) ** 2)
    assert mse_l < 0.95 * mse_u
    # inverse shape, brute-force nearest level over the same span
    inv = np.array([0.0, 1.0, 1.0 + O.LM_RATIO, 2.0 + O.LM_RATIO]) * (2 * O.LM_RATIO + 1) / (2 + O.LM_RATIO)
    g = r.reshape(-1, 128).astype(np.float64)
    mn, mx = g.min(1, keepdims=True), g.max(1, keepdims=True)
    levels = mn[..., None] + (mx - mn)[..., None] / (2 * O.LM_RATIO + 1) * inv
    mse_inv = np.mean(np.min((g[..., None] - levels) ** 2, -1))
    assert mse_inv > mse_u


def test_lloyd_max_constant_group_and_flag_layout():
    r = np.full((1, 128), -0.75, np.float32)
    codes, sc, ze = O.quantize_rows(r, 1.0, lloyd_max=True)
    assert float(sc[0, 0]) == 0.0 and float(ze[0, 0]) == -0.75 and (codes == 0).all()
    # the flag changes the meaning of the codes, not the bytes' layout
    a = O.layout(O.Config(2, 3, 8, 2, 256, 16, 32, 500))
    b = O.layout(O.Config(2, 3, 8, 2, 256, 16, 32, 500, flags=O.FLAG_LLOYD_MAX))
    assert a == b


def test_lloyd_max_decode_equals_library_sdpa_on_exact_rows():
    # S = W = 0: every position is INT2; on Lloyd-Max lattice rows (R = I, clip 1)
    # both K and V are stored exactly, so the decode is plain attention over (K, V)
    B, H, G, D, T = 2, 2, 4, 128, 50
    cfg = O.Config(1, B, H * G, H, D, 0, 0, 64, 1.0, 1.0, flags=O.FLAG_LLOYD_MAX)
    rng = np.random.default_rng(32)
    k = _lm_lattice_rows(rng, (B, T, H, D))
    v = _lm_lattice_rows(rng, (B, T, H, D))
    q = S.to_bf16_values(rng.standard_normal((B, H * G, D)).astype(np.float32))
    I = np.eye(D, dtype=np.float32)
    cache = O.new_cache(cfg)
    O.append(cfg, cache, 0, k, v, [0, 0], I, I)
    lens = [T, 31]
    out, lse = O.decode(cfg, cache, 0, q, lens, I, I)
    for b in range(B):
        Tb = lens[b]
        qt = torch.from_numpy(q[b].astype(np.float64))[:, None, :]
        kt = torch.from_numpy(k[b, :Tb].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        vt = torch.from_numpy(v[b, :Tb].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0].numpy()
        assert np.abs(out[b] - ref).max() < 1e-11 * max(1.0, np.abs(ref).max())
        sc_ = torch.einsum("hd,htd->ht", qt[:, 0], kt) / math.sqrt(D)
        assert np.abs(lse[b] - torch.logsumexp(sc_, -1).numpy()).max() < 1e-11
    # the same cache read with uniform levels is a different (wrong) answer
    plain = O.Config(1, B, H * G, H, D, 0, 0, 64, 1.0, 1.0)
    out_u, _ = O.decode(plain, cache, 0, q, lens, I, I)
    assert np.abs(out_u - out).max() > 1e-2


# --------------------------------------------------------------------------
# R_V calibration: score-weighted V covariance
# --------------------------------------------------------------------------
def test_score_energy_is_the_sum_of_squared_logits():
    # brute force over every (query, key) logit in plain Python
    rng = np.random.default_rng(61)
    q = rng.standard_normal((7, 16))
    k = rng.standard_normal((5, 16))
    w = O.score_energy(q, k)
    for t in range(5):
        tot = 0.0
        for n in range(7):
            tot += sum(float(q[n, i]) * float(k[t, i]) for i in range(16)) ** 2
        assert abs(w[t] - tot) <= 1e-12 * tot


def _rank_hadamard_bitrev(rank, d):
    # R[i, j] = H[rank(i), br(j)] for E = the permutation sending channel i to column rank(i)
    bits = d.bit_length() - 1
    br = [int(format(j, f"0{bits}b")[::-1], 2) for j in range(d)]
    return np.array([[(-1.0) ** bin(int(rank[i]) & br[j]).count("1") / math.sqrt(d) for j in range(d)]
                     for i in range(d)])


@pytest.mark.parametrize("d", [128, 256])
def test_calibrate_rv_diagonal_closed_form_weights_decide_the_order(d):
    # channel i: value rows +-a_i e_i with key e_i; queries sigma_j e_j.  Every
    # weight of channel i is sigma_i^2, so Sigma_V = diag(2 sigma_i^2 a_i^2).  The
    # magnitudes a_i grow with i (the unweighted V covariance ranks channels by
    # i); sigma_i a_i = perm(i) + 1 ranks them by perm instead
    rng = np.random.default_rng(62 + d)
    perm = rng.permutation(d)
    a = 1.0 + np.arange(d) / d
    sig = (perm + 1.0) / a
    Q = np.diag(sig)
    K = np.repeat(np.eye(d), 2, axis=0)
    V = np.repeat(np.diag(a), 2, axis=0) * np.tile([1.0, -1.0], d)[:, None]
    R = O.calibrate_rv(Q, K, V)
    rank = np.empty(d, int)
    rank[np.argsort(-perm, kind="stable")] = np.arange(d)
    assert np.abs(R - _rank_hadamard_bitrev(rank, d)).max() < 1e-12
    # without the weights the order would follow a_i
    assert np.abs(O.calibrate_rk(V) - _rank_hadamard_bitrev(np.arange(d)[::-1], d)).max() < 1e-12


def test_calibrate_rv_reduces_to_the_v_covariance_for_isotropic_queries():
    # Q^T Q = 9 I and unit-norm keys give every key the weight 9: R_V is then the
    # fit of V's own covariance
    d = 128
    rng = np.random.default_rng(63)
    Q = 3.0 * np.eye(d)
    K = rng.standard_normal((900, d))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = S.activations(rng, (900, d), [4, 50, 100], kind="t3")
    assert np.abs(O.calibrate_rv(Q, K, V) - O.calibrate_rk(V)).max() < 1e-9


def test_calibrate_rv_eigen_equation_on_token_by_token_covariance():
    # Sigma_V summed one token at a time from the explicit logit matrix; undoing
    # H P_br (scipy's Hadamard) leaves its eigenvectors, descending and signed
    L = pytest.importorskip("scipy.linalg")
    d = 128
    rng = np.random.default_rng(64)
    ch = [5, 40, 99]
    Q = S.activations(rng, (500, d), ch, kind="t3").astype(np.float64)
    K = S.activations(rng, (400, d), ch, kind="t3").astype(np.float64)
    V = S.activations(rng, (400, d), ch, kind="t3").astype(np.float64)
    logits = Q @ K.T
    sig = np.zeros((d, d))
    for t in range(K.shape[0]):
        sig += float(np.sum(logits[:, t] ** 2)) * np.outer(V[t], V[t])
    R = O.calibrate_rv(Q, K, V)
    bits = d.bit_length() - 1
    P = np.zeros((d, d))
    for i in range(d):
        P[i, int(format(i, f"0{bits}b")[::-1], 2)] = 1.0
    E = R @ P.T @ (L.hadamard(d) / math.sqrt(d)).T
    lam = np.einsum("ij,ij->j", E, sig @ E)
    assert np.abs(sig @ E - E * lam).max() < 1e-9 * lam[0]
    assert np.all(np.diff(lam) <= 1e-9 * lam[0])
    assert np.abs(E.T @ E - np.eye(d)).max() < 1e-12
    piv = np.argmax(np.abs(E), axis=0)
    assert np.all(E[piv, np.arange(d)] > 0)
