"""Quantise-on-append on the GPU is bit-exact with the oracle's block codec.

Page "自研RDNA高併發推論引擎 以AI Max+ 395為範例", §2: the blocked KV mode is
bit-exact at the codec level; q8 blocks are 34 bytes, 4-bit blocks 18 bytes.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

PAIRS = [(wl.FMT_Q8_0, wl.FMT_Q8_0), (wl.FMT_Q4_0, wl.FMT_Q4_0), (wl.FMT_F16, wl.FMT_F16),
         (wl.FMT_Q8_0, wl.FMT_Q4_0), (wl.FMT_Q4_0, wl.FMT_Q8_0)]


def _golden_blocks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "codec_blocks.json")))
    out = []
    for fmt in ("q8_0", "q4_0"):
        for case in g[fmt]:
            xs = case.get("x") or [case["fill"]] * 32
            vals = []
            for s in xs:
                if s == "-0":
                    vals.append(-0.0)
                elif "*2^" in s:
                    a, e = s.split("*2^")
                    vals.append(float(Fraction(int(a)) * Fraction(2) ** int(e)))
                else:
                    vals.append(float(Fraction(s)))
            out.append(np.array(vals, dtype=np.float16))
    return out


def _adversarial(n_tok, hkv, d, seed, golden):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n_tok, hkv, d)).astype(np.float32)
    scale = np.exp2(rng.integers(-24, 8, size=(n_tok, hkv, d // 32, 1))).astype(np.float32)
    x = (x.reshape(n_tok, hkv, d // 32, 32) * scale).astype(np.float16)
    flat = x.reshape(-1, 32)
    flat[::5, 7] = -flat[::5, 2]          # magnitude ties between signs
    flat[::9] = np.float16(0)             # all-zero blocks
    flat[::11, 31] = np.float16(-0.0)
    for i, blk in enumerate(golden):      # the hand-derived blocks, verbatim
        flat[(13 * i + 3) % len(flat)] = blk
    return flat.reshape(n_tok, hkv, d)


@pytest.mark.parametrize("kf,vf", PAIRS)
@pytest.mark.parametrize("d", [64, 128])
def test_append_is_bit_exact(golden_dir, kf, vf, d):
    import torch
    import mixed_attention_quantized_gb300 as mq
    hkv, n_tok, num_pages = 3, 1000, 40
    gold = _golden_blocks(golden_dir)
    k = _adversarial(n_tok, hkv, d, 1, gold)
    v = _adversarial(n_tok, hkv, d, 2, gold[::-1])
    rng = np.random.default_rng(3)
    slots = rng.permutation(num_pages * 32)[:n_tok].astype(np.int32)
    slots[::17] = -1  # padding tokens write nothing
    cache = mq.KVCache.allocate(num_pages, hkv, d, kf, vf, fill=0xA5)
    mq.kv_append_quant(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                       torch.from_numpy(slots).cuda())
    keep = slots >= 0
    sd = torch.from_numpy(slots[keep]).cuda()
    got_k = mq.kv_export_blocks(cache, 0, sd).cpu().numpy()
    got_v = mq.kv_export_blocks(cache, 1, sd).cpu().numpy()
    torch.cuda.synchronize()
    assert mq.device_error(clear=True) == 0
    ref_k = oracle.quantize(kf, k[keep])
    ref_v = oracle.quantize(vf, v[keep])
    assert np.array_equal(got_k, ref_k), np.argwhere(got_k != ref_k)[:5]
    assert np.array_equal(got_v, ref_v), np.argwhere(got_v != ref_v)[:5]
    # slots that no token maps to keep the fill pattern
    used = set(slots[keep].tolist())
    free = np.array(sorted(set(range(num_pages * 32)) - used), dtype=np.int32)[:64]
    untouched = mq.kv_export_blocks(cache, 0, torch.from_numpy(free).cuda()).cpu().numpy()
    assert (untouched == 0xA5).all()


def test_append_plane_layout_matches_the_header():
    """Q8_0 planes: quant [page][head][token][D] int8, scale [page][head][token][D/32] fp16."""
    import torch
    import mixed_attention_quantized_gb300 as mq
    hkv, d, num_pages = 2, 128, 4
    w = wl.custom("layout", 8, hkv, d, wl.FMT_Q8_0, wl.FMT_Q8_0, seed=8, rows=[(wl.ROW_CHUNK, 100, 0)])
    k, v = wl.row_kv(w, 0)
    slots = np.arange(100, dtype=np.int32) + 17
    cache = mq.KVCache.allocate(num_pages, hkv, d, wl.FMT_Q8_0, wl.FMT_Q8_0)
    mq.kv_append_quant(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                       torch.from_numpy(slots).cuda())
    kq = cache.k_quant.cpu().numpy().reshape(num_pages, hkv, 32, d)
    ks = cache.k_scale.cpu().numpy().view(np.uint16).reshape(num_pages, hkv, 32, d // 32)
    ref = oracle.quantize(wl.FMT_Q8_0, k)  # [100, hkv, 4, 34]
    for t in (0, 14, 15, 50, 99):
        s = slots[t]
        for g in range(hkv):
            blocks = ref[t, g]
            assert np.array_equal(kq[s // 32, g, s % 32].view(np.int8), blocks[:, 2:].view(np.int8).ravel())
            assert np.array_equal(ks[s // 32, g, s % 32], blocks[:, :2].copy().view(np.uint16).ravel())


def test_out_of_range_slot_sets_the_device_error_and_is_skipped():
    import torch
    import mixed_attention_quantized_gb300 as mq
    mq.device_error(clear=True)
    cache = mq.KVCache.allocate(2, 1, 64, wl.FMT_Q8_0, wl.FMT_Q8_0, fill=0x5A)
    k = np.ones((2, 1, 64), dtype=np.float16)
    slots = np.array([64, 3], dtype=np.int32)  # 64 == num_pages * 32: out of range
    mq.kv_append_quant(cache, torch.from_numpy(k).cuda(), torch.from_numpy(k).cuda(),
                       torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert mq.device_error(clear=True) & mq.DEVERR_SLOT
    blk = mq.kv_export_blocks(cache, 0, torch.tensor([3], dtype=torch.int32, device="cuda")).cpu().numpy()
    assert np.array_equal(blk, oracle.quantize(wl.FMT_Q8_0, k[1:2]))
    assert mq.device_error(clear=True) == 0
