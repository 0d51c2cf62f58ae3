"""GPU parity of the bfloat16 format (q, K/V and out in bf16, fp32
accumulation) against the f64 oracle.

Tolerance, derived like the fp16 bar: rounding the exact output to bf16 (7
fraction bits) gives a relative error uniform in +-2^-9 per element, a
relative L2 of about 1.1e-3 and, for |out| < 4, an absolute error below
2^-8 = 3.9e-3.  The bar keeps the fp16 bar's headroom over its floor:
relative L2 <= 3e-3, max abs <= 1e-2, per-row relative L2 <= 6e-3.
A context of one position still returns the V row bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS, ROW_REL = 3e-3, 1e-2, 6e-3
DEV = "cuda:0"
BF = torch.bfloat16


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


def check(out, ref, rows=None):
    g = out.float().cpu().numpy().astype(np.float64).reshape(-1, out.shape[-1])
    if rows is not None:
        g = g[rows]
    r = ref.reshape(-1, ref.shape[-1])
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rn = np.linalg.norm(r, axis=1)
    rrel = (np.linalg.norm(g - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert rel <= REL_L2 and np.abs(g - r).max() <= MAX_ABS and rrel <= ROW_REL, (rel, rrel)
    return rel


def run(pkg, w, **kw):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw.setdefault("max_seq_len", w.max_seq_len())
    out = pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                          window=kw.pop("window", w.window), err_flag=err, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert out.dtype == BF
    return out


@pytest.mark.parametrize("name", ["tiny", "llama", "sweep_d64", "sweep_d256", "long_w4096",
                                  "batched"])
def test_bf16_parity(pkg, name):
    w = workloads.make(name, device=DEV, dtype=BF)
    out = run(pkg, w)
    wc = w.to("cpu")
    ref = oracle.decode_attn(wc.q, wc.k_pages, wc.v_pages, wc.page_table, wc.seq_lens, wc.scale,
                             w.window)
    check(out, ref)


@pytest.mark.parametrize("split_min", [0, 1, 100000])
def test_bf16_short_contexts(pkg, split_min):
    base = workloads.make("ctx512_d128", device="cpu", dtype=BF)
    for L in (1, 2, 63, 64, 65, 255, 256, 257, 511):
        w = workloads.Workload(**{**base.__dict__,
                                  "seq_lens": torch.tensor([L], dtype=torch.int32)})
        ref = oracle.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale)
        check(run(pkg, w.to(DEV), split_min=split_min), ref)


def test_bf16_context_one_returns_v_row(pkg):
    lens = [1, 17, 300]
    w = workloads.make_custom("b1", batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                              page_size=16, seq_lens=lens, seed=70, device=DEV, dtype=BF)
    out = run(pkg, w, window=1)
    for b, L in enumerate(lens):
        phys = int(w.page_table[b, (L - 1) // 16])
        for hq in range(8):
            assert torch.equal(out[b, hq], w.v_pages[phys, (L - 1) % 16, hq // 4])


def test_bf16_multi_query_and_fused_append(pkg):
    T, lens = 2, [40, 700, 2]
    w = workloads.make_custom("bm", batch=3, num_q_heads=16, num_kv_heads=4, head_dim=128,
                              page_size=32, seq_lens=lens, seed=71, dtype=BF)
    g = torch.Generator().manual_seed(72)
    q = torch.randn(3, T, 16, 128, generator=g).to(BF)
    kn = torch.randn(3, T, 4, 128, generator=g).to(BF)
    vn = torch.randn(3, T, 4, 128, generator=g).to(BF)
    L = torch.tensor(lens, dtype=torch.int32)
    ok, ov = w.k_pages.clone(), w.v_pages.clone()
    for i in range(T):
        k_np, v_np, _ = oracle.kv_append(kn[:, i].contiguous(), vn[:, i].contiguous(),
                                         L - T + i, w.page_table, ok, ov)
        ok = torch.from_numpy(k_np.view(np.int16)).view(BF).view(ok.shape)
        ov = torch.from_numpy(v_np.view(np.int16)).view(BF).view(ov.shape)
    ref = oracle.decode_attn_multi(q, ok, ov, w.page_table, L, w.scale, 0)
    kp, vp = w.k_pages.to(DEV), w.v_pages.to(DEV)
    out = pkg.decode_attn_append(q.to(DEV), kn.to(DEV), vn.to(DEV), kp, vp,
                                 w.page_table.to(DEV), L.to(DEV), w.scale,
                                 max_seq_len=int(L.max()))
    torch.cuda.synchronize()
    assert torch.equal(kp.cpu(), ok) and torch.equal(vp.cpu(), ov)
    check(out, ref)


def test_bf16_long_context_all_rows(pkg):
    w = workloads.make("long", device=DEV, dtype=BF)
    out = run(pkg, w)
    wc = w.to("cpu")
    ref = oracle.decode_attn(wc.q, wc.k_pages, wc.v_pages, wc.page_table, wc.seq_lens, wc.scale,
                             0)
    check(out, ref)
