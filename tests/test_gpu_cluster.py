"""Cluster plans (DECODE_ATTN_SCHEDULE_CLUSTER: the shards of one (KV head,
sequence) form a thread-block cluster and merge through distributed shared
memory) against the f64 oracle, and bit for bit against the same plan merged
through the workspace (the grid schedule): the two merges share their
arithmetic and shard order."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GRID, CLUSTER = 1, 2
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


def run(pkg, q, w, L, window, max_len, schedule, **kw):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.decode_attn(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window=window,
                          max_seq_len=max_len, err_flag=err, schedule=schedule, **kw)
    torch.cuda.synchronize()
    return out, int(err.item())


def check(out, ref, dtype):
    rel_t, mab_t, row_t = TOL[dtype]
    g = out.float().cpu().numpy().astype(np.float64).reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(r, axis=1)
    assert np.all(g[rn == 0] == 0)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rrel = (np.linalg.norm(g - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert rel <= rel_t and np.abs(g - r).max() <= mab_t and rrel <= row_t, (rel, rrel)


@pytest.mark.parametrize("D,Hq,Hkv,PS,lens,window,T,dtype,chunk", [
    (128, 32, 8, 16, [3060], 0, 1, torch.float16, 384),            # Llama shape, 8 shards
    (64, 32, 8, 16, [3060], 0, 1, torch.float16, 384),             # D = 64, 8 shards
    (256, 16, 4, 16, [3060], 0, 1, torch.bfloat16, 512),           # D = 256
    (128, 64, 8, 64, [9000, 300, 0, 4097], 0, 1, torch.float16, 0),  # short ones: empty shards
    (128, 64, 8, 64, [9000, 2000, 5], 700, 1, torch.float16, 0),   # window
    (128, 16, 4, 32, [2500, 777, 1], 0, 2, torch.float16, 320),    # T = 2, 8 query rows
    (256, 16, 4, 16, [3060], 0, 1, torch.float16, 0),              # planner: 16 shards, 64 CTAs
    (128, 16, 2, 16, [4000, 300], 0, 2, torch.bfloat16, 512),      # T = 2, G = 8: 16 rows
    (64, 8, 8, 16, [1000, 1000], 0, 1, torch.float16, 128),        # G = 1, 8 shards
])
def test_cluster_parity_and_bits(pkg, D, Hq, Hkv, PS, lens, window, T, dtype, chunk):
    w = workloads.make_custom("c", batch=len(lens), num_q_heads=Hq, num_kv_heads=Hkv,
                              head_dim=D, page_size=PS, seq_lens=[max(L, 1) for L in lens],
                              seed=41 + D + Hq, decoy_pages=3, dtype=dtype)
    L = torch.tensor(lens, dtype=torch.int32)
    g = torch.Generator().manual_seed(42 + D)
    if T > 1:
        q = torch.randn(len(lens), T, Hq, D, generator=g).to(dtype)
        ref = oracle.decode_attn_multi(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window)
    else:
        q = w.q
        ref = oracle.decode_attn(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window)
    wd, qd, Ld = w.to(DEV), q.to(DEV), L.to(DEV)
    max_len = max(lens)
    params = pkg.make_params(qd, wd.k_pages, wd.page_table, w.scale, window, max_len, 0, 0,
                             chunk, CLUSTER)
    plan = pkg.decode_attn_make_plan(params,
                                     torch.cuda.get_device_properties(DEV).multi_processor_count)
    assert plan.cluster == plan.max_shards and 2 <= plan.cluster <= 16, plan.as_dict()
    out_c, err_c = run(pkg, qd, wd, Ld, window, max_len, CLUSTER, force_chunk=chunk)
    out_g, err_g = run(pkg, qd, wd, Ld, window, max_len, GRID, force_chunk=chunk)
    assert err_c == 0 and err_g == 0
    check(out_c, ref, dtype)
    assert torch.equal(out_c, out_g)
    again, _ = run(pkg, qd, wd, Ld, window, max_len, CLUSTER, force_chunk=chunk)
    assert torch.equal(out_c, again)


def test_cluster_split_then_combine_equals(pkg):
    """decode_attn_combine re-merges the partials a cluster launch also left
    in the workspace: the same bits as the cluster merge (the head_dim-256
    sweep shape: 16 shards in clusters of 16)."""
    w = workloads.make("sweep_d256", device=DEV)
    params = pkg.make_params(w.q, w.k_pages, w.page_table, w.scale, 0, w.max_seq_len(), 0, 0,
                             0, CLUSTER)
    out, ws = pkg.decode_attn_split(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens,
                                    w.scale, max_seq_len=w.max_seq_len(), schedule=CLUSTER)
    torch.cuda.synchronize()
    fused = out.clone()
    out.zero_()
    pkg.decode_attn_combine(params, w.seq_lens, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, fused)


def test_cluster_bad_rows_are_zero(pkg):
    lens = [500, 0, 300, 400, 600, 2000]
    w = workloads.make_custom("cb", batch=6, num_q_heads=8, num_kv_heads=2, head_dim=128,
                              page_size=16, seq_lens=[max(L, 1) for L in lens], seed=86,
                              device=DEV)
    cap = w.page_table.shape[1] * 16
    table = w.page_table.clone()
    table[2, 3] = w.k_pages.shape[0] + 5
    table[3, 1] = -7
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    seq[4] = cap + 1
    w2 = workloads.Workload(**{**w.__dict__, "page_table": table, "seq_lens": seq})
    out, err = run(pkg, w2.q, w2, seq, 0, cap, CLUSTER, force_chunk=512)
    assert err & pkg.DEV_BAD_PAGE and err & pkg.DEV_BAD_LEN
    assert torch.all(out[1:5] == 0)
    ref = oracle.decode_attn(w2.q.cpu(), w2.k_pages.cpu(), w2.v_pages.cpu(), table.cpu(),
                             seq.cpu(), w.scale, 0, rows=np.r_[0:8, 40:48])
    check(out.view(-1, 128)[np.r_[0:8, 40:48]], ref, torch.float16)


def test_cluster_stall_with_empty_shards_reports_timeout_and_recovers(pkg):
    """A cluster plan whose clusters hold empty shards (a 300-token and an
    empty sequence beside a 9000-token one), with every CTA's first-stage
    barrier made to expect 64 bytes more than its copies bring (the library's
    DECODE_ATTN_TEST_STALL_TX hook): the empty shards reach the exchange at
    once and must still wait for their partners, whose consumers give up
    after about 2 s.  The call ends by itself with DECODE_ATTN_DEV_TIMEOUT and
    zero rows; the next call is again bit-identical to the workspace merge and
    within tolerance of the oracle."""
    import os
    lens = [9000, 300, 0, 4097]
    w = workloads.make_custom("cs", batch=4, num_q_heads=64, num_kv_heads=8, head_dim=128,
                              page_size=64, seq_lens=[max(L, 1) for L in lens], seed=87,
                              decoy_pages=3)
    L = torch.tensor(lens, dtype=torch.int32)
    ref = oracle.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, L, w.scale, 0)
    wd, Ld = w.to(DEV), L.to(DEV)
    params = pkg.make_params(wd.q, wd.k_pages, wd.page_table, w.scale, 0, 9000, 0, 0, 0,
                             CLUSTER)
    plan = pkg.decode_attn_make_plan(params,
                                     torch.cuda.get_device_properties(DEV).multi_processor_count)
    assert plan.cluster == plan.max_shards >= 2, plan.as_dict()
    os.environ["DECODE_ATTN_TEST_STALL_TX"] = "64"
    try:
        out, err = run(pkg, wd.q, wd, Ld, 0, 9000, CLUSTER)
    finally:
        del os.environ["DECODE_ATTN_TEST_STALL_TX"]
    assert err & pkg.DEV_TIMEOUT
    assert torch.all(out == 0)
    out_c, err_c = run(pkg, wd.q, wd, Ld, 0, 9000, CLUSTER)
    out_g, err_g = run(pkg, wd.q, wd, Ld, 0, 9000, GRID)
    assert err_c == 0 and err_g == 0
    assert torch.equal(out_c, out_g)
    check(out_c, ref, torch.float16)
