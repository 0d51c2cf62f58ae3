"""GPU parity of the persistent, balanced schedule (one CTA per resident
slot, equal ranges of the flattened (sequence, KV head, tile) list, partial
units merged by their last CTA) against the f64 oracle, across the features
the grid schedule has: mixed lengths, windows, T query positions, bf16, the
fused append, invalid inputs, run-to-run bits."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
P = 2  # SCHEDULE_PERSISTENT
TOL = {torch.float16: (5e-4, 2e-3, 1e-3), torch.bfloat16: (3e-3, 1e-2, 6e-3)}


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
    rel_t, mab_t, row_t = TOL[out.dtype]
    g = out.float().cpu().numpy().astype(np.float64).reshape(-1, out.shape[-1])
    if rows is not None:
        g = g[rows]
    r = ref.reshape(-1, ref.shape[-1])
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rn = np.linalg.norm(r, axis=1)
    rrel = (np.linalg.norm(g - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert np.all(g[rn == 0] == 0)
    assert rel <= rel_t and np.abs(g - r).max() <= mab_t and rrel <= row_t, (rel, rrel)


def run(pkg, w, q=None, **kw):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw.setdefault("max_seq_len", w.max_seq_len())
    kw.setdefault("schedule", P)
    out = pkg.decode_attn(w.q if q is None else q, w.k_pages, w.v_pages, w.page_table,
                          w.seq_lens, w.scale, window=kw.pop("window", w.window), err_flag=err,
                          **kw)
    torch.cuda.synchronize()
    return out, int(err.item())


def ref_of(w, window=None, rows=None):
    wc = w.to("cpu")
    return oracle.decode_attn(wc.q, wc.k_pages, wc.v_pages, wc.page_table, wc.seq_lens, wc.scale,
                              w.window if window is None else window, rows=rows)


@pytest.mark.parametrize("name", ["batched", "long_w4096", "llama", "sweep_d64", "sweep_d256",
                                  "tiny"])
def test_persistent_parity(pkg, name):
    w = workloads.make(name, device=DEV)
    out, err = run(pkg, w)
    assert err == 0
    check(out, ref_of(w))


def test_persistent_long_sampled_rows(pkg):
    w = workloads.make("long", device=DEV)
    out, err = run(pkg, w)
    assert err == 0
    Hq = w.num_q_heads
    rows = np.array([b * Hq + hq for b in range(w.batch) for hq in (0, 13, 26, 39, 52, 63)])
    check(out, ref_of(w, rows=rows), rows=rows)


@pytest.mark.parametrize("PS,D,window", [(16, 128, 0), (8, 64, 0), (32, 256, 90), (64, 128, 0)])
def test_many_short_sequences(pkg, PS, D, window):
    """A thousand sequences of 0..300 positions: CTA ranges cut units at
    arbitrary tiles and hold many units each."""
    g = torch.Generator().manual_seed(80 + PS)
    lens = torch.randint(0, 301, (1000,), generator=g)
    lens[::97] = 0
    w = workloads.make_custom("many", batch=1000, num_q_heads=8, num_kv_heads=2, head_dim=D,
                              page_size=PS, seq_lens=torch.clamp(lens, min=1), seed=81,
                              device=DEV)
    w.seq_lens = lens.to(torch.int32).to(DEV)
    out, err = run(pkg, w, window=window, max_seq_len=300)
    assert err == 0
    check(out, ref_of(w, window=window))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_persistent_multi_query(pkg, dtype):
    T, lens = 4, [3, 700, 2500, 64, 1]
    w = workloads.make_custom("mq", batch=5, num_q_heads=16, num_kv_heads=4, head_dim=128,
                              page_size=16, seq_lens=lens, seed=82, dtype=dtype)
    g = torch.Generator().manual_seed(83)
    q = torch.randn(5, T, 16, 128, generator=g).to(dtype)
    L = torch.tensor(lens, dtype=torch.int32)
    ref = oracle.decode_attn_multi(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, 0)
    wd = w.to(DEV)
    out, err = run(pkg, wd, q=q.to(DEV))
    assert err == 0
    check(out, ref)


def test_persistent_fused_append(pkg):
    T, lens = 2, [130, 4097, 1, 65]
    w = workloads.make_custom("pa", batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              page_size=64, seq_lens=lens, seed=84)
    g = torch.Generator().manual_seed(85)
    q = torch.randn(4, T, 32, 128, generator=g).half()
    kn = torch.randn(4, T, 8, 128, generator=g).half()
    vn = torch.randn(4, T, 8, 128, generator=g).half()
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
                                 max_seq_len=int(L.max()), schedule=P)
    torch.cuda.synchronize()
    assert torch.equal(kp.cpu(), ok) and torch.equal(vp.cpu(), ov)
    check(out, ref)


def test_persistent_errors_zero_only_bad_rows(pkg):
    lens = [500, 0, 300, 400, 600, 2000]
    w = workloads.make_custom("pe", batch=6, num_q_heads=8, num_kv_heads=2, head_dim=128,
                              page_size=16, seq_lens=[max(L, 1) for L in lens], seed=86,
                              device=DEV)
    cap = w.page_table.shape[1] * 16
    table = w.page_table.clone()
    table[2, 3] = w.k_pages.shape[0] + 5
    table[3, 1] = -7
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    seq[4] = cap + 1
    w2 = workloads.Workload(**{**w.__dict__, "page_table": table, "seq_lens": seq})
    out, err = run(pkg, w2, max_seq_len=cap)
    assert err & pkg.DEV_BAD_PAGE and err & pkg.DEV_BAD_LEN
    assert torch.all(out[1:5] == 0)
    ok_rows = np.r_[0:8, 40:48]
    check(out.view(-1, 128)[ok_rows], ref_of(w2, rows=ok_rows))


def test_persistent_run_to_run_bitwise_and_agrees_with_grid(pkg):
    w = workloads.make("batched", device=DEV)
    first, _ = run(pkg, w)
    for _ in range(3):
        again, _ = run(pkg, w)
        assert torch.equal(first, again)
    grid, _ = run(pkg, w, schedule=1)
    g = grid.float().cpu().numpy().astype(np.float64)
    check(first, g)


def test_persistent_with_static_scratch_and_graph(pkg):
    w = workloads.make("long_w4096", device=DEV)
    ref, _ = run(pkg, w)
    out = pkg.decode_attn_static_scratch(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens,
                                         w.scale, window=w.window, max_seq_len=w.max_seq_len(),
                                         schedule=P)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    out2 = torch.empty_like(w.q)
    max_len = w.max_seq_len()  # host value, read before the capture
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                        window=w.window, out=out2, max_seq_len=max_len, schedule=P)
    gr.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2, ref)
