"""hswa_decode_noalloc: the decode entry point for callers that cannot give
the library a workspace (their device memory is owned by someone else, or
they may not allocate at all). Its scratch is a fixed array inside the
library, so the caller passes only inputs and outputs.

Checked through the C ABI against hswa_decode (which takes a caller-owned
workspace) on two calls in a row, so that a second call that starts from the
first call's leftover scratch still gives the right result. This file sorts
last so that a run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest
import torch

import hswa_workloads as wl
import hybrid_sliding_window_dual_gb300 as H
from scenario import Scenario, TOL


def test_noalloc_rejects_batches_beyond_its_limit():
    cfg = H.Config(window=128, page_size=64, n_q_heads=64, n_kv_heads=8, head_dim=128, dtype=H.HSWA_DTYPE_BF16,
                   full_pages=8, swa_pages=8, max_seqs=4, max_pages_per_seq=4)
    pool = H.hswa_pool_create(cfg)
    layer = H.Layer(kind=H.HSWA_KIND_FULL, window=128, k_pool=256, v_pool=256)
    too_many = H.lib.hswa_decode_noalloc(pool, layer, 256, 256, 256, 256, 16385, 1.0, None)
    assert too_many == H.HSWA_ERR_INVALID_ARG
    H.hswa_pool_destroy(pool)


@pytest.mark.gpu
@pytest.mark.parametrize("kinds", [(wl.KIND_FULL, wl.KIND_SWA)])
def test_noalloc_decode_matches_workspace_decode_twice(kinds):
    cached = [0, 1, 63, 64, 65, 300, 2000, 9000, 129, 5]
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, cached, layer_kinds=kinds, seed=41)
    B = len(cached)
    full_slots, swa_slots = sc.reserve(range(B), [1] * B)
    sc.sess.sync()
    for layer, slots in ((0, full_slots), (1, swa_slots)):
        q = sc.to_dev(sc.gen((B, 64, 128), 10 + layer))
        kn = sc.to_dev(sc.gen((B, 8, 128), 20 + layer))
        vn = sc.to_dev(sc.gen((B, 8, 128), 30 + layer))
        sc.sess.append(layer, kn, vn, torch.as_tensor(slots, device="cuda"))
        ref = torch.empty_like(q)
        sc.sess.decode(layer, q, ref, B, sc.scale)  # caller-owned workspace
        assert sc.sess.check() == 0
        for _ in range(2):
            out = torch.full_like(q, float("nan"))
            H.hswa_decode_noalloc(sc.sess.pool, sc.sess.layers[layer], q, out, sc.sess.bt(layer),
                                  sc.sess.d_seq_len, B, sc.scale, sc.sess.stream)
            assert sc.sess.check() == 0
            assert H.hswa_last_kernel() == "decode_mma_bf16_d128"
            err = (out.float() - ref.float()).abs().max().item()
            assert err <= TOL[wl.DTYPE_BF16], err
