"""Pins for the FP8 KV-cache part of the oracle (no GPU).

* the E4M3 codec against torch's float8_e4m3fn (a library routine): every
  code decoded, random in-range values encoded, ties to even, saturation;
* the per-tile quantizer: the largest element of a tile maps to +-448, a
  zero tile gets scale 1, and every value comes back within half an E4M3
  step of itself;
* FP8 attention against torch scaled_dot_product_attention in float64 on the
  dequantized dense data (Full and windows), with the transposed V page;
* with unit scales and values that bf16 holds exactly, FP8 attention equals
  the bf16 oracle bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from test_oracle import sdpa_reference


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = fp8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000) * 50, rng.standard_normal(20000) * 0.01,
                        [0.0, -0.0, 448.0, -448.0, 1e-12, -1e-12]]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), ref)


def test_e4m3_ties_round_to_even_and_saturate():
    # 1.0625 lies halfway between 1.0 (code 0x38) and 1.125 (0x39): the even code wins
    assert fp8.e4m3_encode(np.array([1.0625]))[0] == 0x38
    assert fp8.e4m3_encode(np.array([1.1875]))[0] == 0x3A  # between 0x39 and 0x3a
    big = fp8.e4m3_encode(np.array([449.0, 1e9, -1e9]))
    assert list(big) == [0x7E, 0x7E, 0xFE]


@pytest.mark.parametrize("seed", [0, 1])
def test_quantize_tiles_bounds(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((5, 3, 256)) * rng.uniform(0.01, 100, (5, 3, 1))).astype(np.float32)
    x[2, 1, :128] = 0.0
    codes, scales = fp8.quantize_tiles(x)
    assert codes.shape == x.shape and scales.shape == (5, 3, 2)
    assert scales[2, 1, 0] == 1.0 and (codes[2, 1, :128] == 0).all()
    t = np.abs(x.reshape(5, 3, 2, 128))
    arg = t.argmax(-1)
    top = np.take_along_axis(codes.reshape(5, 3, 2, 128), arg[..., None], -1)[..., 0]
    nonzero = t.max(-1) > 0
    assert (top[nonzero] & 0x7F == 0x7E).all()
    back = fp8.dequantize_tiles(codes, scales)
    # half a step of E4M3 (3 mantissa bits) relative, or half the subnormal step
    err = np.abs(back - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.repeat(scales, 128, -1) * 2.0 ** -10)
    assert (err <= bound * (1 + 1e-6)).all()


def random_fp8_case(seed, S=3, hq=8, hkv=2, d=128, P=4, lmax=29):
    """Dense fp32 K/V, quantized per (token, head) tile, placed in pages."""
    rng = np.random.default_rng(seed)
    n_lp = -(-lmax // P)
    perm = rng.permutation(S * n_lp + 3)[:S * n_lp].reshape(S, n_lp).astype(np.int32)
    pages = int(perm.max()) + 1
    k = rng.standard_normal((S, hkv, lmax, d)).astype(np.float32)
    v = rng.standard_normal((S, hkv, lmax, d)).astype(np.float32)
    kc = np.zeros((pages, hkv, P, d), np.uint8)
    vc = np.zeros((pages, hkv, d, P), np.uint8)
    ks = np.ones((pages, hkv, P, d // 128), np.float32)
    vs = np.ones_like(ks)
    kq, ksc = fp8.quantize_tiles(k)
    vq, vsc = fp8.quantize_tiles(v)
    for s in range(S):
        for j in range(lmax):
            pg, r = perm[s, j // P], j % P
            kc[pg, :, r, :] = kq[s, :, j, :]
            ks[pg, :, r, :] = ksc[s, :, j, :]
            vc[pg, :, :, r] = vq[s, :, j, :]
            vs[pg, :, r, :] = vsc[s, :, j, :]
    kd = fp8.dequantize_tiles(kq, ksc)
    vd = fp8.dequantize_tiles(vq, vsc)
    return kd, vd, (kc, ks, vc, vs), perm


def test_fp8_attention_matches_sdpa_on_dequantized_data():
    hq, hkv, d = 8, 2, 128
    kd, vd, (kc, ks, vc, vs), bt = random_fp8_case(3, hq=hq, hkv=hkv, d=d)
    rng = np.random.default_rng(5)
    worst = 0.0
    for window in (0, 1, 6, 64):
        for s in range(kd.shape[0]):
            pos = np.array([0, 3, 4, 17, 28], np.int64)
            q = rng.standard_normal((len(pos), hq, d)).astype(np.float32)
            got = oracle.attention_fp8(q, kc, ks, vc, vs, bt, np.full(len(pos), s), pos, window, 1 / math.sqrt(d))
            ref = sdpa_reference(q, kd.astype(np.float64), vd.astype(np.float64), s, pos, window,
                                 1 / math.sqrt(d), hq)
            worst = max(worst, float(np.abs(got - ref).max()))
    assert worst < 1e-12, worst


def test_fp8_attention_equals_bf16_oracle_on_exact_values():
    """Codes with unit scales are values bf16 holds exactly: both oracles agree bit for bit."""
    rng = np.random.default_rng(7)
    pages, hkv, P, d = 6, 1, 4, 128
    kc = rng.integers(0, 0x7E, (pages, hkv, P, d)).astype(np.uint8) | (rng.integers(0, 2, (pages, hkv, P, d)) << 7).astype(np.uint8)
    vc = rng.integers(0, 0x7E, (pages, hkv, d, P)).astype(np.uint8)
    ones = np.ones((pages, hkv, P, 1), np.float32)
    kf = fp8.e4m3_decode(kc).astype(np.float32) / 64
    vf = np.transpose(fp8.e4m3_decode(vc), (0, 1, 3, 2)).astype(np.float32)
    bt = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    q = rng.standard_normal((2, 4, d)).astype(np.float32)
    a = oracle.attention_fp8(q, kc, ones / 64, vc, ones, bt, [0, 1], [10, 7], 0, 0.1)
    b = oracle.attention(q, np.ascontiguousarray(kf), np.ascontiguousarray(vf), bt, [0, 1], [10, 7], 0, 0.1)
    assert np.array_equal(a, b)


def test_append_fp8_writes_rows_and_transposed_values():
    P, hkv, d = 4, 2, 128
    kc = np.zeros((3, hkv, P, d), np.uint8)
    vc = np.zeros((3, hkv, d, P), np.uint8)
    ks = np.zeros((3, hkv, P, 1), np.float32)
    vs = np.zeros_like(ks)
    new = np.random.default_rng(1).standard_normal((2, hkv, d)).astype(np.float32)
    oracle.append_kv_fp8(kc, ks, vc, vs, new, -new, [5, 11])
    q, s = fp8.quantize_tiles(new)
    assert np.array_equal(kc[1, :, 1, :], q[0]) and np.array_equal(kc[2, :, 3, :], q[1])
    assert np.array_equal(ks[1, :, 1, :], s[0])
    qv, sv = fp8.quantize_tiles(-new)
    assert np.array_equal(vc[2, :, :, 3], qv[1]) and np.array_equal(vs[2, :, 3, :], sv[1])


FP8_MUTATIONS = {
    "v_not_transposed": ("v_codes[(b * head_dim + c) * page_size + row]", "v_codes[(b * page_size + row) * head_dim + c]"),
    "k_scale_of_next_row": ("k_scale[(b * page_size + row) * tiles + c / 128]",
                            "k_scale[(b * page_size + (row + 1) % page_size) * tiles + c / 128]"),
    "subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "exponent_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTATIONS))
def test_fp8_pins_catch_planted_mistake(name, tmp_path):
    import os
    import subprocess
    import sys
    src = open(os.path.join(os.path.dirname(oracle.__file__), "hswa_oracle.c")).read()
    old, new = FP8_MUTATIONS[name]
    assert src.count(old) >= 1, name
    (tmp_path / "mut.c").write_text(src.replace(old, new))
    so = tmp_path / "mut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", str(tmp_path / "mut.c"), "-o", str(so),
                           "-lm"])
    here = os.path.dirname(__file__)
    code = ("import sys; sys.path[:0] = [%r, %r]; import math, numpy as np, oracle, test_oracle_fp8 as t\n"
            "from test_oracle import sdpa_reference\n"
            "lib = oracle.load_library(%r)\n"
            "kd, vd, (kc, ks, vc, vs), bt = t.random_fp8_case(3)\n"
            "q = np.random.default_rng(5).standard_normal((5, 8, 128)).astype(np.float32)\n"
            "pos = np.array([0, 3, 4, 17, 28])\n"
            "worst = 0.0\n"
            "for s in range(3):\n"
            "    got = oracle.attention_fp8(q, kc, ks, vc, vs, bt, np.full(5, s), pos, 0, 0.1, lib=lib)\n"
            "    ref = sdpa_reference(q, kd, vd, s, pos, 0, 0.1, 8)\n"
            "    worst = max(worst, float(np.abs(got - ref).max()))\n"
            "print('FAILED' if not worst < 1e-12 else 'ok')\n" % (os.path.dirname(here), here, str(so)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 or "FAILED" in r.stdout, r.stdout


# ------------------------------------------------------------- FP8 transfer
def fp8_pools(seed, pages=12, hkv=2, P=4):
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 0x7F, (pages, hkv, P, 128)).astype(np.uint8) | (rng.integers(0, 2, (pages, hkv, P, 128)) << 7).astype(np.uint8)
    vc = rng.integers(0, 0x7F, (pages, hkv, 128, P)).astype(np.uint8)
    ks = rng.uniform(0.001, 0.01, (pages, hkv, P, 1)).astype(np.float32)
    vs = rng.uniform(0.001, 0.01, (pages, hkv, P, 1)).astype(np.float32)
    return kc, ks, vc, vs


def test_fp8_pack_is_the_dequantized_window():
    """Dequantizing the packed codes with the packed scales gives the pool's
    dequantized K and V at each window token (V read back from the
    transposed pages), sequence by sequence."""
    kc, ks, vc, vs = fp8_pools(3)
    bt = np.array([[5, 2, 9, -1], [0, 7, 11, 3]], np.int32)  # W = 6: sequence 0 needs pages 1, 2 only
    lens, W, hkv, P = [11, 14], 6, 2, 4
    bt[0, 3] = -1
    buf = oracle.swa_pack_fp8(kc, ks, vc, vs, bt, lens, W)
    n, off = oracle.swa_window_counts(lens, W)
    assert buf.size == int(off[-1]) * 2 * hkv * 132
    kd = fp8.dequantize_tiles(kc, ks)                                  # [pages][Hkv][P][d]
    vd = fp8.dequantize_tiles(np.transpose(vc, (0, 1, 3, 2)), vs)      # token rows
    for s, L in enumerate(lens):
        ns, base = int(n[s]), int(off[s]) * 2 * hkv * 132
        c = hkv * ns * 128
        kb = buf[base:base + c].reshape(hkv, ns, 128)
        vb = buf[base + c:base + 2 * c].reshape(hkv, ns, 128)
        kss = buf[base + 2 * c:base + 2 * c + 4 * hkv * ns].view(np.float32).reshape(hkv, ns)
        vss = buf[base + 2 * c + 4 * hkv * ns:base + 2 * c + 8 * hkv * ns].view(np.float32).reshape(hkv, ns)
        for i, t in enumerate(range(L - ns, L)):
            pg, r = bt[s, t // P], t % P
            assert np.array_equal(fp8.e4m3_decode(kb[:, i]) * kss[:, i, None], kd[pg, :, r])
            assert np.array_equal(fp8.e4m3_decode(vb[:, i]) * vss[:, i, None], vd[pg, :, r])


def test_fp8_unpack_restores_the_window_into_fresh_pages():
    kc, ks, vc, vs = fp8_pools(4)
    bt = np.array([[1, 4, 6], [2, 8, 10]], np.int32)
    lens, W = [9, 12], 5
    buf = oracle.swa_pack_fp8(kc, ks, vc, vs, bt, lens, W)
    fresh = [np.zeros_like(x) for x in (kc, ks, vc, vs)]
    bt2 = np.array([[0, 3, 5], [7, 9, 11]], np.int32)  # other pages
    oracle.swa_unpack_fp8(buf, fresh[0], fresh[1], fresh[2], fresh[3], bt2, lens, W)
    assert np.array_equal(oracle.swa_pack_fp8(*fresh, bt2, lens, W), buf)
    # only window tokens were written: position 3 of sequence 0 (page 0, row 3) stays zero
    assert not fresh[0][0, :, 3].any() and not fresh[2][0, :, :, 3].any()
