"""GPU parity for several query positions per sequence (T new tokens, each
attending causally up to itself, e.g. speculative verification or a suffix
prefill over the paged cache) against the f64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS, ROW_REL = 5e-4, 2e-3, 1e-3
DEV = "cuda:0"


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_gqa_decode_06_gb300 import build
    build.build()
    oracle.build()
    import paged_gqa_decode_06_gb300 as p
    p.load_library()
    return p


def case(seed, lens, T, Hq, Hkv, D, PS):
    w = workloads.make_custom("m", batch=len(lens), num_q_heads=Hq, num_kv_heads=Hkv,
                              head_dim=D, page_size=PS, seq_lens=[max(L, 1) for L in lens],
                              seed=seed, decoy_pages=3)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(len(lens), T, Hq, D, generator=g).half()
    L = torch.tensor(lens, dtype=torch.int32)
    return w, q, L


def check(out, ref):
    g = out.float().cpu().numpy().astype(np.float64).reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rn = np.linalg.norm(r, axis=1)
    rrel = (np.linalg.norm(g - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    zero_rows = rn == 0
    assert np.all(g[zero_rows] == 0)
    assert rel <= REL_L2 and np.abs(g - r).max() <= MAX_ABS and rrel <= ROW_REL, (rel, rrel)


@pytest.mark.parametrize("T,Hq,Hkv,D,PS", [
    (2, 16, 4, 128, 16),   # 8 query rows per KV head
    (4, 16, 4, 128, 64),   # 16 rows
    (2, 32, 4, 64, 32),    # G = 8: 16 rows
    (16, 8, 8, 128, 16),   # G = 1: 16 rows
    (3, 12, 4, 256, 16),   # 9 rows padded to 16
])
@pytest.mark.parametrize("window", [0, 200])
@pytest.mark.parametrize("split_min", [0, 1, 100000])
def test_multi_query_parity(pkg, T, Hq, Hkv, D, PS, window, split_min):
    lens = [T - 1, T, 300, 2500, 5]
    w, q, L = case(50 + T, lens, T, Hq, Hkv, D, PS)
    ref = oracle.decode_attn_multi(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    wd = w.to(DEV)
    out = pkg.decode_attn(q.to(DEV), wd.k_pages, wd.v_pages, wd.page_table, L.to(DEV),
                          w.scale, window=window, max_seq_len=int(L.max()), err_flag=err,
                          split_min=split_min)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and out.shape == q.shape
    check(out, ref)


def test_one_query_as_4d_equals_3d(pkg):
    w = workloads.make("llama", device=DEV)
    a = pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                        max_seq_len=w.max_seq_len())
    b = pkg.decode_attn(w.q[:, None].contiguous(), w.k_pages, w.v_pages, w.page_table,
                        w.seq_lens, w.scale, max_seq_len=w.max_seq_len())
    torch.cuda.synchronize()
    assert torch.equal(a, b[:, 0])


@pytest.mark.parametrize("chunk", [0, 64])
def test_fused_append_of_several_tokens(pkg, chunk):
    """T new rows written at the last T positions inside the split kernel,
    also when they straddle two shards (64-token shards)."""
    T, Hq, Hkv, D, PS = 4, 16, 4, 128, 16
    lens = [130, 66, 4, 1000]   # 130: positions 126..129 cross the 128 boundary
    w = workloads.make_custom("ma", batch=4, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              page_size=PS, seq_lens=lens, seed=60, decoy_pages=2)
    g = torch.Generator().manual_seed(61)
    q = torch.randn(4, T, Hq, D, generator=g).half()
    kn = torch.randn(4, T, Hkv, D, generator=g).half()
    vn = torch.randn(4, T, Hkv, D, generator=g).half()
    L = torch.tensor(lens, dtype=torch.int32)
    ok, ov = w.k_pages.clone(), w.v_pages.clone()
    for i in range(T):
        k_np, v_np, _ = oracle.kv_append(kn[:, i].contiguous(), vn[:, i].contiguous(),
                                         L - T + i, w.page_table, ok, ov)
        ok = torch.from_numpy(k_np.view(np.int16)).view(torch.float16).view(ok.shape)
        ov = torch.from_numpy(v_np.view(np.int16)).view(torch.float16).view(ov.shape)
    ref = oracle.decode_attn_multi(q, ok, ov, w.page_table, L, w.scale, 0)
    kp, vp = w.k_pages.to(DEV), w.v_pages.to(DEV)
    out = pkg.decode_attn_append(q.to(DEV), kn.to(DEV), vn.to(DEV), kp, vp,
                                 w.page_table.to(DEV), L.to(DEV), w.scale,
                                 max_seq_len=int(L.max()), force_chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(kp.cpu(), ok) and torch.equal(vp.cpu(), ov)
    check(out, ref)
