"""The all-heads schedule (DECODE_ATTN_SCHEDULE_ALL_HEADS: persistent CTAs
that stream 16-position slices of all 8 KV heads per stage, one consumer
warp per head, work items (sequence, shard) from an atomic counter) against
the f64 oracle; bit-identical run to run and to decode_attn_combine's
re-merge of its partials; its error rows, its timeout path, the append path
it takes (separate append kernel, then attention), and the batched
workload on it."""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
AUTO, GRID, ALL_HEADS = 0, 1, 4
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


def check(out, ref, dtype):
    rel_t, mab_t, row_t = TOL[dtype]
    g = out.float().cpu().numpy().astype(np.float64).reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(r, axis=1)
    assert np.all(np.isfinite(g))
    assert np.all(g[rn == 0] == 0)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rrel = (np.linalg.norm(g - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert rel <= rel_t and np.abs(g - r).max() <= mab_t and rrel <= row_t, (rel, rrel)


def plan_of(pkg, q, w, window, max_len, chunk, schedule):
    params = pkg.make_params(q, w.k_pages, w.page_table, w.scale, window, max_len, 0, 0, chunk,
                             schedule)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    return params, pkg.decode_attn_make_plan(params, sms)


def run(pkg, w, L, window, max_len, chunk, schedule=ALL_HEADS, ws=None):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window=window,
                          max_seq_len=max_len, err_flag=err, schedule=schedule,
                          force_chunk=chunk, workspace=ws)
    torch.cuda.synchronize()
    return out, int(err.item())


MIXED = [0, 1, 15, 16, 17, 255, 256, 257, 511, 512, 513, 1000, 3000, 8192, 4097, 63]


@pytest.mark.parametrize("D,Hq,PS,lens,window,dtype,chunk", [
    (128, 32, 16, MIXED, 0, torch.float16, 0),          # the planner's chunk (512)
    (128, 32, 16, MIXED, 0, torch.float16, 256),
    (128, 32, 16, MIXED, 0, torch.float16, 1024),
    (64, 32, 32, MIXED, 0, torch.bfloat16, 0),          # D = 64: 6 stages
    (128, 32, 64, MIXED, 0, torch.bfloat16, 512),
    (128, 8, 128, MIXED, 0, torch.float16, 384),        # G = 1
    (128, 64, 16, MIXED, 0, torch.float16, 0),          # G = 8
    (128, 32, 16, MIXED, 700, torch.float16, 0),        # window, unaligned starts
    (64, 16, 16, [5, 9000, 333, 2], 1000, torch.float16, 320),
])
def test_all_heads_parity_and_bits(pkg, D, Hq, PS, lens, window, dtype, chunk):
    w = workloads.make_custom("ah", batch=len(lens), num_q_heads=Hq, num_kv_heads=8,
                              head_dim=D, page_size=PS, seq_lens=[max(L, 1) for L in lens],
                              seed=500 + D + Hq + PS + window, decoy_pages=5, dtype=dtype)
    L = torch.tensor(lens, dtype=torch.int32)
    ref = oracle.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window)
    wd, Ld = w.to(DEV), L.to(DEV)
    max_len = max(lens)
    _, plan = plan_of(pkg, wd.q, wd, window, max_len, chunk, ALL_HEADS)
    assert plan.all_heads == 1 and plan.split == 1, plan.as_dict()
    out, err = run(pkg, wd, Ld, window, max_len, chunk)
    assert err == 0
    check(out, ref, dtype)
    again, err = run(pkg, wd, Ld, window, max_len, chunk)
    assert err == 0 and torch.equal(out, again)
    # decode_attn_combine re-merges the partials the launch left: same bits
    params, _ = plan_of(pkg, wd.q, wd, window, max_len, chunk, ALL_HEADS)
    part, ws = pkg.decode_attn_split(wd.q, wd.k_pages, wd.v_pages, wd.page_table, Ld, w.scale,
                                     window=window, max_seq_len=max_len, force_chunk=chunk,
                                     schedule=ALL_HEADS)
    torch.cuda.synchronize()
    assert torch.equal(part, out)
    part.zero_()
    pkg.decode_attn_combine(params, Ld, part, ws)
    torch.cuda.synchronize()
    assert torch.equal(part, out)


def test_all_heads_bad_rows(pkg):
    """A bad page id, a length past the table and an empty sequence: the
    error bits, zero rows for those sequences, the others exact."""
    lens = [3000, 900, 0, 1500, 700, 20]
    w = workloads.make_custom("ahbad", batch=6, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              page_size=16, seq_lens=[max(L, 1) for L in lens], seed=611,
                              device=DEV)
    cap = w.page_table.shape[1] * 16
    table = w.page_table.clone()
    table[1, 40] = w.k_pages.shape[0] + 3     # inside sequence 1's second shard of 512
    table[4, 2] = -2                          # sequence 4, first of its two shards
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    seq[3] = cap + 5
    w2 = workloads.Workload(**{**w.__dict__, "page_table": table, "seq_lens": seq})
    out, err = run(pkg, w2, seq, 0, cap, 512)
    assert err & pkg.DEV_BAD_PAGE and err & pkg.DEV_BAD_LEN
    for b in (1, 2, 3, 4):
        assert torch.all(out[b] == 0), b
    keep = np.r_[0:32, 160:192]
    ref = oracle.decode_attn(w.q.cpu(), w.k_pages.cpu(), w.v_pages.cpu(), w.page_table.cpu(),
                             torch.tensor(lens, dtype=torch.int32), w.scale, 0, rows=keep)
    check(out.view(-1, 128)[keep], ref, torch.float16)
    # a clean call right after, on the same workspace defaults, is exact
    out, err = run(pkg, w, w.seq_lens, 0, cap, 512)
    assert err == 0


def test_all_heads_batched_matches_oracle(pkg):
    """The batched workload (64 sequences of U[1, 8192] positions, 32/8
    heads, page 16) on the all-heads schedule and on the planner's own
    pick, against the oracle."""
    w = workloads.make("batched", device=DEV)
    max_len = w.max_seq_len()
    _, plan = plan_of(pkg, w.q, w, 0, max_len, 0, AUTO)
    assert plan.all_heads == 0, plan.as_dict()
    out, err = run(pkg, w, w.seq_lens, 0, max_len, 0, schedule=ALL_HEADS)
    assert err == 0
    wc = w.to("cpu")
    rows = np.arange(0, 64 * 32, 5)
    ref = oracle.decode_attn(wc.q, wc.k_pages, wc.v_pages, wc.page_table, wc.seq_lens, w.scale, 0,
                             rows=rows)
    check(out.view(-1, 128)[rows], ref, torch.float16)
    grid, err = run(pkg, w, w.seq_lens, 0, max_len, 0, schedule=AUTO)
    assert err == 0
    check(grid.view(-1, 128)[rows], ref, torch.float16)


def test_all_heads_append_path(pkg):
    """decode_attn_append on an all-heads plan: the rows land bit-exact (the
    append kernel runs first) and the attention matches the oracle."""
    lens = [0, 1, 300, 4000, 2047]
    B, Hq, D, PS = len(lens), 32, 128, 16
    w = workloads.make_custom("aha", batch=B, num_q_heads=Hq, num_kv_heads=8, head_dim=D,
                              page_size=PS, seq_lens=[L + 1 for L in lens], seed=77,
                              decoy_pages=3)
    g = torch.Generator().manual_seed(78)
    kn = torch.randn(B, 8, D, generator=g).half()
    vn = torch.randn(B, 8, D, generator=g).half()
    L_after = torch.tensor([L + 1 if L > 0 else 0 for L in lens], dtype=torch.int32)
    pos = L_after - 1
    ref_k, ref_v, _ = oracle.kv_append(kn, vn, pos, w.page_table, w.k_pages, w.v_pages)
    ref = oracle.decode_attn(w.q, ref_k, ref_v, w.page_table, L_after, w.scale, 0)
    kp, vp = w.k_pages.to(DEV), w.v_pages.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.decode_attn_append(w.q.to(DEV), kn.to(DEV), vn.to(DEV), kp, vp,
                                 w.page_table.to(DEV), L_after.to(DEV), w.scale,
                                 max_seq_len=int(L_after.max()), err_flag=err,
                                 schedule=ALL_HEADS)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    u16 = lambda t: torch.from_numpy(np.ascontiguousarray(t).view(np.int16)).view(torch.float16)
    assert torch.equal(kp.cpu(), u16(ref_k).view(kp.shape))
    assert torch.equal(vp.cpu(), u16(ref_v).view(vp.shape))
    check(out, ref, torch.float16)


def test_all_heads_stall_reports_timeout_and_recovers(pkg):
    """Every CTA's first stage expects 64 bytes more than it brings (the
    DECODE_ATTN_TEST_STALL_TX hook): the call ends by itself with
    DECODE_ATTN_DEV_TIMEOUT, and after the workspace is cleared the next
    call is exact."""
    lens = [3000, 2500, 4000, 1000] * 4
    w = workloads.make_custom("ahstall", batch=len(lens), num_q_heads=32, num_kv_heads=8,
                              head_dim=128, page_size=16, seq_lens=lens, seed=88, device=DEV)
    params, plan = plan_of(pkg, w.q, w, 0, max(lens), 512, ALL_HEADS)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=DEV)
    os.environ["DECODE_ATTN_TEST_STALL_TX"] = "64"
    try:
        _, err = run(pkg, w, w.seq_lens, 0, max(lens), 512, ws=ws)
    finally:
        del os.environ["DECODE_ATTN_TEST_STALL_TX"]
    assert err & pkg.DEV_TIMEOUT
    pkg.decode_attn_workspace_clear(params, ws)
    out, err = run(pkg, w, w.seq_lens, 0, max(lens), 512, ws=ws)
    assert err == 0
    wc = w.to("cpu")
    ref = oracle.decode_attn(wc.q, wc.k_pages, wc.v_pages, wc.page_table, wc.seq_lens, w.scale, 0)
    check(out, ref, torch.float16)
