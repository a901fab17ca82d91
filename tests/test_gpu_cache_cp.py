"""GPU parity of the context-parallel slot mapping and the KV-cache write
against the oracle (bit-exact: both are integer / copy work), and of a
context-parallel decode on simulated ranks: each rank's slots, cache write and
attention over the keys it owns, merged by LSE, against the oracle's attention
over the whole sequence."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu_helpers import LSE_ATOL, max_errors, oracle_rows
from oracle import swa_oracle as O
import paged_sliding_window_swa_gb300 as swa

pytestmark = pytest.mark.gpu


def _requests(rng, n_req, max_len, bs, spare):
    lens = rng.integers(1, max_len + 1, size=n_req)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pos = np.concatenate([np.arange(int(n)) for n in lens]).astype(np.int64)
    pages = -(-int(lens.max()) // bs) + spare
    bt = rng.permutation(n_req * pages).reshape(n_req, pages).astype(np.int32)
    return qsl, pos, bt


@pytest.mark.parametrize("seed", range(16))
def test_slot_mapping_cp_matches_oracle(seed):
    rng = np.random.default_rng(700 + seed)
    bs = int(rng.choice([16, 32, 64]))
    world = int(rng.choice([1, 2, 3, 4, 8]))
    kvb = bs * int(rng.choice([1, 2, 4]))
    divisors = [d for d in range(1, kvb + 1) if kvb % d == 0]
    inter = int(rng.choice(divisors))
    rank = int(rng.integers(0, world))
    qsl, pos, bt = _requests(rng, int(rng.integers(1, 6)), 3000, bs, spare=4)
    if seed % 4 == 0 and len(pos) > 2:
        pos[1] = -5                                   # a bad position
    T = int(qsl[-1])
    maxn = T + int(rng.integers(0, 20))
    exp, bad = O.slot_mapping_cp(qsl, pos, bt, bs, maxn, kvb, world, rank, inter)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = swa.swa_slot_mapping_cp(torch.as_tensor(qsl, device="cuda"), torch.as_tensor(pos, device="cuda"),
                                  torch.as_tensor(bt, device="cuda"), bs, maxn, kv_cache_block_size=kvb,
                                  cp_world_size=world, cp_rank=rank, cp_interleave=inter, err=err)
    assert np.array_equal(got.cpu().numpy(), exp)
    torch.cuda.synchronize()
    assert bool(err.item() & 0x02) == bool(bad)


def test_slot_mapping_cp_section_3_3_example():
    bt = torch.tensor([[7, 3, 11, 5]], dtype=torch.int32, device="cuda")
    pos = torch.arange(512, dtype=torch.int64, device="cuda")
    qsl = torch.tensor([0, 512], dtype=torch.int32, device="cuda")
    r0 = swa.swa_slot_mapping_cp(qsl, pos, bt, 128, 512, kv_cache_block_size=128, cp_world_size=2, cp_rank=0,
                                 cp_interleave=128).cpu().numpy()
    exp0 = np.full(512, -1)
    exp0[0:128] = 7 * 128 + np.arange(128)
    exp0[256:384] = 3 * 128 + np.arange(128)
    assert np.array_equal(r0, exp0)


@pytest.mark.parametrize("dtype,D,hkv", [("bf16", 128, 8), ("bf16", 256, 8), ("fp32", 64, 2), ("bf16", 72, 3)])
def test_kv_cache_write_matches_oracle(dtype, D, hkv):
    rng = np.random.default_rng(D + hkv)
    bs = 16
    qsl, pos, bt = _requests(rng, 4, 700, bs, spare=6)
    T = int(qsl[-1])
    slots, _ = O.slot_mapping(qsl, pos, bt, bs, T, T + 7)
    slots = slots.astype(np.int64)
    nblocks = int(bt.max()) + 1
    slots[3] = nblocks * bs + 9                       # past the cache: reported, not written
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kc = torch.randn((nblocks, bs, hkv, D), device="cuda").to(tdt)
    vc = torch.randn((nblocks, bs, hkv, D), device="cuda").to(tdt)
    kn = torch.randn((T + 7, hkv, D), device="cuda").to(tdt)
    vn = torch.randn((T + 7, hkv, D), device="cuda").to(tdt)
    ek, ev, bad = O.kv_cache_write(kn.float().cpu().numpy(), vn.float().cpu().numpy(), slots,
                                   kc.float().cpu().numpy(), vc.float().cpu().numpy())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    swa.swa_kv_cache_write(kn, vn, torch.as_tensor(slots.astype(np.int32), device="cuda"), kc, vc, err=err)
    assert np.array_equal(kc.float().cpu().numpy(), ek) and np.array_equal(vc.float().cpu().numpy(), ev)
    torch.cuda.synchronize()
    assert bad == [3] and err.item() == 0x80


def test_cache_written_through_slots_gives_the_same_attention():
    """The Gemma-like layout's caches rebuilt from dense per-token K/V through
    swa_slot_mapping + swa_kv_cache_write: attention is bit-identical."""
    lay = W.random_small(77, head_dim=256, group=2, max_seqs=3, max_ctx=600, max_q=400, with_ranges=True)
    q, k, v = W.make_tensors(lay, device="cuda")
    d = W.device_layout(lay, "cuda")
    B, hkv, D = lay.block_size, lay.num_heads_kv, lay.head_dim
    # every key of every sequence, in order, as "new" tokens at positions 0..seq_len-1
    toks_k, toks_v, pos, qsl = [], [], [], [0]
    for s in range(lay.num_seqs):
        L = int(lay.seq_lens[s])
        for p in range(L):
            blk = int(lay.block_table[s][p // B])
            toks_k.append(k[blk, p % B])
            toks_v.append(v[blk, p % B])
        pos.append(torch.arange(L, dtype=torch.int64, device="cuda"))
        qsl.append(qsl[-1] + L)
    kn, vn = torch.stack(toks_k), torch.stack(toks_v)
    slots = swa.swa_slot_mapping(torch.tensor(qsl, dtype=torch.int32, device="cuda"), torch.cat(pos),
                                 d["block_table"], B, len(toks_k))
    k2, v2 = torch.zeros_like(k), torch.zeros_like(v)
    swa.swa_kv_cache_write(kn, vn, slots, k2, v2)

    def run(kc, vc):
        return swa.swa_mm_paged_attention(q, kc, vc, d["block_table"], d["query_start_loc"], d["seq_lens"],
                                          mm_ranges=d["mm_ranges"], max_query_len=lay.max_query_len,
                                          window=lay.window, causal=lay.causal, scale=lay.scale)
    o1, l1 = run(k, v)
    o2, l2 = run(k2, v2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("world,inter", [(2, 16), (4, 64), (3, 32), (8, 16)])
def test_rank_split_decode_merges_to_full_attention(world, inter):
    """Context-parallel decode with the cache interleaved over `world` simulated
    ranks: each rank maps its slots, writes the keys it owns and attends over
    them (its query sees every local key); lse_combine over the ranks gives
    the attention over the whole sequence."""
    rng = np.random.default_rng(world * 1000 + inter)
    bs, hq, hkv, D = 16, 8, 2, 128
    lens = rng.integers(300, 4000, size=5)
    S = len(lens)
    kv = [(torch.randn((int(n), hkv, D), device="cuda").to(torch.bfloat16),
           torch.randn((int(n), hkv, D), device="cuda").to(torch.bfloat16)) for n in lens]
    q = torch.randn((S, hq, D), device="cuda").to(torch.bfloat16)
    scale = D ** -0.5
    pages = int(-(-lens.max() // bs)) + 2
    ctx_qsl = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    positions = torch.cat([torch.arange(int(n), dtype=torch.int64, device="cuda") for n in lens])
    kn = torch.cat([a for a, _ in kv])
    vn = torch.cat([b for _, b in kv])
    kvb = int(np.lcm(bs, inter))
    q_qsl = torch.arange(S + 1, dtype=torch.int32, device="cuda")
    po = torch.empty((world, S, hq, D), dtype=torch.bfloat16, device="cuda")
    pl = torch.empty((world, S, hq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(world):
        bt_r = torch.as_tensor(rng.permutation(S * pages).reshape(S, pages).astype(np.int32), device="cuda")
        slots = swa.swa_slot_mapping_cp(ctx_qsl, positions, bt_r, bs, int(lens.sum()), kv_cache_block_size=kvb,
                                        cp_world_size=world, cp_rank=r, cp_interleave=inter, err=err)
        kc = torch.zeros((S * pages, bs, hkv, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        swa.swa_kv_cache_write(kn, vn, slots, kc, vc, err=err)
        n_local = torch.stack([(slots[int(ctx_qsl[s]):int(ctx_qsl[s + 1])] >= 0).sum() for s in range(S)]).to(torch.int32)
        swa.swa_mm_paged_attention(q, kc, vc, bt_r, q_qsl, n_local, max_query_len=1, window=0, causal=False,
                                   scale=scale, out=po[r], lse=pl[r], err=err)
    mo, ml = swa.lse_combine(po, pl)
    torch.cuda.synchronize()
    assert err.item() == 0
    # the oracle: one query per sequence at its last position over all keys
    kc_full = np.zeros((S * pages, bs, hkv, D))
    vc_full = np.zeros_like(kc_full)
    bt_full = rng.permutation(S * pages).reshape(S, pages)
    for s in range(S):
        ks, vs = kv[s][0].float().cpu().numpy(), kv[s][1].float().cpu().numpy()
        for p in range(int(lens[s])):
            kc_full[bt_full[s, p // bs], p % bs] = ks[p]
            vc_full[bt_full[s, p // bs], p % bs] = vs[p]
    ro, rl = O.attention(q.float().cpu().numpy(), kc_full, vc_full, bt_full, np.arange(S + 1), lens, None, 0,
                         True, scale)
    rows = [(s, h) for s in range(S) for h in range(hq)]
    e_out, e_lse = max_errors(mo, ml, ro, rl, rows)
    assert e_out <= 2e-2 and e_lse <= LSE_ATOL
