"""hswa_decode_noalloc: the decode entry point for callers that cannot give
the library a workspace (their device memory is owned by someone else, or
they may not allocate at all). Its scratch is a fixed array inside the
library, so the caller passes only inputs and outputs.

Checked through the C ABI against hswa_decode (which takes a caller-owned
workspace) on two calls in a row per layer, each with its own query: both
calls run the same kernels on the same partition, so the outputs must be
identical bit for bit, and a second call that read the first call's leftover
scratch would show. Cases: bf16 pools, FP8 pools (whose decode kernel keeps
more CTAs per SM, so its partials sit closest to the array's end) and a batch
of 3000 short sequences (whose per-sequence descriptors push the partials to
a large offset). This file sorts last so that a run stopping at the first
failure has run everything else.
"""
import math

import numpy as np
import pytest
import torch

import hswa_workloads as wl
import hybrid_sliding_window_dual_gb300 as H
from scenario import Scenario


def test_noalloc_rejects_batches_beyond_its_limit():
    cfg = H.Config(window=128, page_size=64, n_q_heads=64, n_kv_heads=8, head_dim=128, dtype=H.HSWA_DTYPE_BF16,
                   full_pages=8, swa_pages=8, max_seqs=4, max_pages_per_seq=4)
    pool = H.hswa_pool_create(cfg)
    layer = H.Layer(kind=H.HSWA_KIND_FULL, window=128, k_pool=256, v_pool=256)
    too_many = H.lib.hswa_decode_noalloc(pool, layer, 256, 256, 256, 256, 16385, 1.0, None)
    assert too_many == H.HSWA_ERR_INVALID_ARG
    H.hswa_pool_destroy(pool)


def twice_against_workspace_decode(sess, layers, B, make_q, scale, kernel):
    """Per layer: two no-allocation calls in a row with different queries,
    each equal bit for bit to hswa_decode on a caller-owned workspace."""
    for layer in layers:
        for call in range(2):
            q = make_q(layer, call)
            ref = torch.empty_like(q)
            sess.decode(layer, q, ref, B, scale)
            assert sess.check() == 0
            out = torch.full_like(q, float("nan"))
            H.hswa_decode_noalloc(sess.pool, sess.layers[layer], q, out, sess.bt(layer), sess.d_seq_len, B, scale,
                                  sess.stream)
            assert sess.check() == 0
            assert H.hswa_last_kernel() == kernel
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (layer, call)


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_twice():
    cached = [0, 1, 63, 64, 65, 300, 2000, 9000, 129, 5]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=41)
    B = len(cached)
    full_slots, swa_slots = sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    for layer, slots in ((0, full_slots), (1, swa_slots)):
        kn = sc.to_dev(sc.gen((B, 8, 128), 20 + layer))
        vn = sc.to_dev(sc.gen((B, 8, 128), 30 + layer))
        sc.sess.append(layer, kn, vn, torch.as_tensor(slots, device="cuda"))
    twice_against_workspace_decode(sc.sess, (0, 1), B, lambda ly, c: sc.to_dev(sc.gen((B, 64, 128), 10 + 2 * ly + c)),
                                   sc.scale, "decode_mma_bf16_d128")


@pytest.mark.gpu
def test_noalloc_decode_large_batch_of_short_sequences():
    rng = np.random.default_rng(42)
    cached = [int(x) for x in rng.integers(0, 300, size=3000)]
    B = len(cached)
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, seed=42, swa_pages=5 * B + 16)
    sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    twice_against_workspace_decode(sc.sess, (0, 1), B, lambda ly, c: sc.to_dev(sc.gen((B, 64, 128), 50 + 2 * ly + c)),
                                   sc.scale, "decode_mma_bf16_d128")


@pytest.mark.gpu
def test_noalloc_decode_fp8_pools():
    from test_gpu_fp8 import Fp8Case, HQ, D
    cached = [0, 1, 63, 64, 65, 127, 128, 700, 3000, 9000, 20000]
    c = Fp8Case(cached, seed=43)
    B = c.B
    c.sess.reserve(range(B), [1] * B)
    c.sess.sync()
    twice_against_workspace_decode(c.sess, (0, 1), B,
                                   lambda ly, call: wl.normal((B, HQ, D), 60 + 2 * ly + call, wl.DTYPE_BF16).cuda(),
                                   1 / math.sqrt(D), "decode_mma_fp8_d128")
