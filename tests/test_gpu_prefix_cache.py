"""GPU parity of neo_write_prefix_cache against the oracle (a byte copy, so
bit-exact), and a chunked block-causal prefill through the written cache."""

import numpy as np
import pytest
import torch

import oracle as O
from attention_neo_qknorm_gb300 import neo
from helpers import SCALE, assert_bf16_close, f64

pytestmark = pytest.mark.gpu


def _case(lens, N, n_new, Hkv=2, dtype=torch.bfloat16, seed=0, extra=7):
    g = torch.Generator().manual_seed(seed)
    total = int(sum(lens))
    k_old = torch.randn(total, Hkv, 128, generator=g).to(dtype)
    v_old = torch.randn(total, Hkv, 128, generator=g).to(dtype)
    k_new = torch.randn(len(lens), N, Hkv, 128, generator=g).to(dtype)
    v_new = torch.randn(len(lens), N, Hkv, 128, generator=g).to(dtype)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = np.asarray(n_new, np.int32)
    cap = total + int(n.sum()) + extra
    return k_old, v_old, cu, k_new, v_new, n, cap


def _run(k_old, v_old, cu, k_new, v_new, n, cap, use_n=True):
    d = "cuda"
    B, N, Hkv, _ = k_new.shape
    k_out = torch.full((cap, Hkv, 128), 7.0, dtype=k_new.dtype, device=d)
    v_out = torch.full_like(k_out, 7.0)
    cu_out = torch.full((B + 1,), -1, dtype=torch.int32, device=d)
    neo.neo_write_prefix_cache(k_old.to(d) if len(k_old) else None, v_old.to(d) if len(v_old) else None,
                               torch.from_numpy(cu).to(d), k_new.to(d), v_new.to(d), k_out, v_out, cu_out,
                               n_new=torch.from_numpy(n).to(d) if use_n else None)
    return k_out.cpu(), v_out.cpu(), cu_out.cpu().numpy()


@pytest.mark.parametrize("lens,N,n_new,dtype", [
    ((200, 77, 0), 50, (50, 0, 13), torch.bfloat16),    # ragged old rows, ragged chunks, an empty chunk
    ((0, 0), 33, (33, 1), torch.bfloat16),              # empty caches: a first prefill chunk
    ((5,), 16, (16,), torch.float32),                   # fp32 rows
    ((300, 1, 2, 3), 129, (129, 128, 0, 64), torch.bfloat16),
])
def test_cache_write_is_bit_exact(gpu_lib, lens, N, n_new, dtype):
    k_old, v_old, cu, k_new, v_new, n, cap = _case(lens, N, n_new, dtype=dtype)
    k, v, cu_out = _run(k_old, v_old, cu, k_new, v_new, n, cap)
    rk, rv, rcu = O.write_prefix_cache(k_old.numpy() if dtype == torch.float32 else f64(k_old),
                                       v_old.numpy() if dtype == torch.float32 else f64(v_old), cu,
                                       f64(k_new), f64(v_new), n)
    used = int(rcu[-1])
    assert np.array_equal(cu_out, rcu)
    assert np.array_equal(f64(k[:used]), np.asarray(rk, np.float64))
    assert np.array_equal(f64(v[:used]), np.asarray(rv, np.float64))
    assert torch.all(k[used:] == 7.0) and torch.all(v[used:] == 7.0)   # nothing past the packed rows


def test_cache_write_without_counts_appends_whole_chunks(gpu_lib):
    k_old, v_old, cu, k_new, v_new, n, cap = _case((10, 20), 8, (8, 8))
    k, v, cu_out = _run(k_old, v_old, cu, k_new, v_new, n, cap, use_n=False)
    rk, _, rcu = O.write_prefix_cache(f64(k_old), f64(v_old), cu, f64(k_new), f64(v_new), n)
    assert np.array_equal(cu_out, rcu) and np.array_equal(f64(k[:int(rcu[-1])]), rk)


def test_cache_append_in_place_for_one_sequence(gpu_lib):
    g = torch.Generator().manual_seed(5)
    cap, L, N = 300, 120, 70
    k_cache = torch.randn(cap, 2, 128, generator=g).to(torch.bfloat16).cuda()
    v_cache = torch.randn(cap, 2, 128, generator=g).to(torch.bfloat16).cuda()
    before_k, before_v = k_cache.clone(), v_cache.clone()
    k_new = torch.randn(1, N, 2, 128, generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn(1, N, 2, 128, generator=g).to(torch.bfloat16).cuda()
    cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    cu_out = torch.zeros(2, dtype=torch.int32, device="cuda")
    neo.neo_write_prefix_cache(k_cache[:L], v_cache[:L], cu, k_new, v_new, k_cache, v_cache, cu_out)
    assert cu_out.tolist() == [0, L + N]
    assert torch.equal(k_cache[:L], before_k[:L]) and torch.equal(k_cache[L:L + N], k_new[0])
    assert torch.equal(v_cache[L:L + N], v_new[0]) and torch.equal(k_cache[L + N:], before_k[L + N:])


def test_cache_write_bad_counts_set_the_device_error(gpu_lib):
    k_old, v_old, cu, k_new, v_new, n, cap = _case((4, 4), 8, (8, 8))
    neo.neo_get_device_error()
    _run(k_old, v_old, cu, k_new, v_new, np.array([9, 1], np.int32), cap)       # n above N
    st, word = neo.neo_get_device_error()
    assert word & neo.NEO_DEVERR_BAD_PREFIX
    _run(k_old, v_old, cu, k_new, v_new, np.array([8, 8], np.int32), cap - 8)   # beyond capacity
    st, word = neo.neo_get_device_error()
    assert word & neo.NEO_DEVERR_BAD_PREFIX
    _run(k_old, v_old, cu, k_new, v_new, n, cap)
    assert neo.neo_get_device_error() == (neo.NEO_OK, 0)


def test_chunked_prefill_through_the_cache(gpu_lib):
    """Two sequences prefilled in two chunks each: chunk 1 with block-causal
    attention over itself, its keys/values written to the cache, chunk 2 over
    [cache ; itself]; chunk 2's output matches the oracle's one-pass prefill
    of the whole sequences (the image block straddles the chunk boundary)."""
    segs = [[("text", 0, 40), ("image", 40, 8, 8), ("text", 41, 30)],     # 134 tokens
            [("text", 0, 10), ("image", 10, 12, 10), ("text", 11, 4)]]    # 134 tokens
    S, c, Hq, Hkv = 134, 60, 8, 2
    T = np.stack([O.positions(s)[0] for s in segs]).astype(np.int32)
    g = torch.Generator().manual_seed(9)
    q = torch.randn(2, S, Hq, 128, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(2, S, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(2, S, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    Td = torch.from_numpy(T).cuda()
    zero = torch.zeros(3, dtype=torch.int32, device="cuda")
    out1 = torch.empty(2, c, Hq, 128, dtype=torch.bfloat16, device="cuda")
    neo.neo_gen_attention(q[:, :c].contiguous(), None, None, k[:, :c].contiguous(), v[:, :c].contiguous(), zero, 0,
                          out1, scale=SCALE, mask_mode=neo.NEO_MASK_BLOCK_CAUSAL,
                          t_img=Td[:, :c].contiguous().view(-1))
    kc = torch.empty(2 * c, Hkv, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    cu = torch.empty(3, dtype=torch.int32, device="cuda")
    neo.neo_write_prefix_cache(None, None, zero, k[:, :c].contiguous(), v[:, :c].contiguous(), kc, vc, cu)
    tc = Td[:, :c].contiguous().view(-1)      # the cache's temporal indexes, packed like its rows
    out2 = torch.empty(2, S - c, Hq, 128, dtype=torch.bfloat16, device="cuda")
    neo.neo_gen_attention(q[:, c:].contiguous(), kc, vc, k[:, c:].contiguous(), v[:, c:].contiguous(), cu, c, out2,
                          scale=SCALE, mask_mode=neo.NEO_MASK_BLOCK_CAUSAL, t_prefix=tc,
                          t_img=Td[:, c:].contiguous().view(-1))
    empty = np.zeros((0, Hkv, 128))
    qh, kh, vh = f64(q.cpu()), f64(k.cpu()), f64(v.cpu())
    ref, _ = O.gen_attention(qh, empty, empty, kh, vh, [0, 0, 0], SCALE, mask_mode=1,
                             t_prefix=np.zeros(0, np.int32), t_img=T)
    # chunk 1 sees only its own keys (its image queries cannot see the block's
    # rows in chunk 2); chunk 2 sees everything before it, so it equals the
    # one-pass prefill's rows
    ref1, _ = O.gen_attention(qh[:, :c], empty, empty, kh[:, :c], vh[:, :c], [0, 0, 0], SCALE, mask_mode=1,
                              t_prefix=np.zeros(0, np.int32), t_img=T[:, :c])
    assert_bf16_close(f64(out1.cpu()), ref1, "chunk 1")
    assert_bf16_close(f64(out2.cpu()), ref[:, c:], "chunk 2 through the cache")


def test_cache_write_bench_shape(gpu_lib):
    """The append the bench times: caches of 300 / 777 / 1500 / 2048 rows plus
    512-token chunks, 8 KV heads, bf16 (54.7 MB moved)."""
    k_old, v_old, cu, k_new, v_new, n, cap = _case((300, 777, 1500, 2048), 512, (512, 512, 512, 512), Hkv=8,
                                                   seed=21, extra=0)
    k, v, cu_out = _run(k_old, v_old, cu, k_new, v_new, n, cap)
    rk, rv, rcu = O.write_prefix_cache(f64(k_old), f64(v_old), cu, f64(k_new), f64(v_new), n)
    assert np.array_equal(cu_out, rcu)
    assert np.array_equal(f64(k), rk) and np.array_equal(f64(v), rv)
