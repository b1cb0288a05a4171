"""Paged-KV decode (fa_fwd_paged): the same tile update on keys gathered page
by page through a block table.  Held bit for bit to fa_fwd on the same keys
laid out contiguously ("FlashAttention forward in C", section 5), and to the
oracle within the bf16 tolerance for ragged batches."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import compare, oracle_attention

pytestmark = pytest.mark.gpu

BF = torch.bfloat16
DEV = torch.device("cuda", 0)


def _paged_cache(k, v, lens, page_size, seed):
    """Scatter sequences k/v [B, Hkv, Tk, d] into shuffled pages of
    [num_pages, page_size, Hkv, d]; returns caches and the block table."""
    B, Hkv, Tk, d = k.shape
    blocks = [-(-int(L) // page_size) for L in lens]
    max_blocks = max(1, max(blocks))
    total = sum(blocks) + 3  # a few unused pages
    perm = torch.randperm(total, generator=torch.Generator().manual_seed(seed))
    kc = torch.zeros((total, page_size, Hkv, d), dtype=k.dtype)
    vc = torch.zeros_like(kc)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for j in range(blocks[b]):
            page = int(perm[nxt]); nxt += 1
            table[b, j] = page
            lo, hi = j * page_size, min((j + 1) * page_size, int(lens[b]))
            kc[page, :hi - lo] = k[b, :, lo:hi].transpose(0, 1)
            vc[page, :hi - lo] = v[b, :, lo:hi].transpose(0, 1)
    return kc.to(DEV), vc.to(DEV), table.to(DEV), total


@pytest.mark.parametrize("page_size", [16, 64, 128, 256])
def test_paged_bitwise_equals_contiguous(page_size):
    B, Hq, Hkv, Tq, L, d = 3, 16, 8, 1, 3000, 128
    q, k, v = workloads.qkv(80 + page_size, B, Hq, Hkv, Tq, L, d, BF)
    lens = [L] * B
    kc, vc, table, npages = _paged_cache(k, v, lens, page_size, 81)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = fa.paged_attention(q.to(DEV), kc, vc, table, sl, L, scale=d ** -0.5)
    oc, lc = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), scale=d ** -0.5, q_offset=L - Tq, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, oc) and torch.equal(lse, lc)


def test_paged_ragged_batch_vs_oracle():
    B, Hq, Hkv, Tq, d = 5, 8, 2, 1, 64
    lens = [1, 127, 128, 129, 4000]
    L = max(lens)
    q, k, v = workloads.qkv(82, B, Hq, Hkv, Tq, L, d, BF)
    kc, vc, table, _ = _paged_cache(k, v, lens, 32, 83)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = fa.paged_attention(q.to(DEV), kc, vc, table, sl, L, scale=0.125)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    for b, Lb in enumerate(lens):
        eo, el = oracle_attention(q[b:b + 1], k[b:b + 1, :, :Lb], v[b:b + 1, :, :Lb], scale=0.125,
                                  q_offset=Lb - Tq, causal=True)
        compare(o[b:b + 1], lse[b:b + 1], eo, el, BF, f"paged ragged b={b} L={Lb}")


def test_paged_multi_token_sinks_window():
    B, Hq, Hkv, Tq, d = 2, 32, 4, 4, 128
    lens = [2600, 900]
    L = max(lens)
    q, k, v = workloads.qkv(84, B, Hq, Hkv, Tq, L, d, BF)
    z = workloads.sinks(85, Hq)
    kc, vc, table, _ = _paged_cache(k, v, lens, 64, 86)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = fa.paged_attention(q.to(DEV), kc, vc, table, sl, L, scale=d ** -0.5, window=700, sinks=z.to(DEV))
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    for b, Lb in enumerate(lens):
        eo, el = oracle_attention(q[b:b + 1], k[b:b + 1, :, :Lb], v[b:b + 1, :, :Lb], scale=d ** -0.5,
                                  q_offset=Lb - Tq, causal=True, window=700, sinks=z)
        compare(o[b:b + 1], lse[b:b + 1], eo, el, BF, f"paged window/sinks b={b}")


def test_paged_empty_sequence():
    # a sequence with no keys yet: o = 0 and lse = -inf (the sink logit with sinks)
    B, Hq, Hkv, Tq, d = 2, 4, 2, 1, 64
    lens = [0, 300]
    q, k, v = workloads.qkv(87, B, Hq, Hkv, Tq, 300, d, BF)
    kc, vc, table, _ = _paged_cache(k, v, lens, 16, 88)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o, lse = fa.paged_attention(q.to(DEV), kc, vc, table, sl, 300, scale=0.125)
    torch.cuda.synchronize()
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    eo, el = oracle_attention(q[1:2], k[1:2], v[1:2], scale=0.125, q_offset=299, causal=True)
    compare(o[1:2].cpu(), lse[1:2].cpu(), eo, el, BF, "paged second sequence")
