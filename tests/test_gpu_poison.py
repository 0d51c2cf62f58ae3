"""Positions a step does not attend never reach its output, whatever they
hold.  The kernels load whole TMA boxes (up to a page or 64 positions), so the
tail of a sequence's last page, the positions before a sliding window's start
and, for shards sized for the longest sequence, page-table entries past a
sequence's length can be fetched; the pages define the step over the attended
positions only.  Here those places hold NaN or Inf (and every unused
page-table entry is a VALID id of a poisoned page): the output must match the
f64 oracle on clean data, and the same inputs with finite values there bit for
bit, on every kernel path (single pass, grid, cluster, shallow ring,
CUDA-core variant)."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
AUTO, GRID, CLUSTER = 0, 1, 2
V_AUTO, V_SIMT = 0, 1
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


def attended_start(L, window, T):
    """First position any of the T queries attends (the window's reading:
    the last `window` positions up to each query's own position)."""
    first_end = L - T + 1
    return first_end - window if window > 0 and first_end > window else 0


def poisoned(w, lens, window, T, fill, n_poison=5):
    """`n_poison` extra pages of `fill`; every page-table entry past a
    sequence's pages points at one of them; the positions of its used pages
    before its attended start and past its length hold `fill`."""
    P, PS = w.k_pages.shape[0], w.k_pages.shape[1]
    extra = torch.full((n_poison,) + tuple(w.k_pages.shape[1:]), fill, dtype=w.k_pages.dtype)
    k = torch.cat([w.k_pages, extra])
    v = torch.cat([w.v_pages, extra])
    table = w.page_table.clone()
    for b, L in enumerate(lens):
        need = (L + PS - 1) // PS
        for j in range(need, table.shape[1]):
            table[b, j] = P + (b + j) % n_poison
        if L % PS:
            last = int(table[b, L // PS])
            k[last, L % PS:] = fill
            v[last, L % PS:] = fill
        start = attended_start(L, window, T) if L > 0 else 0
        for pos in range(0, start, PS):
            page, n = int(table[b, pos // PS]), min(PS, start - pos)
            k[page, :n] = fill
            v[page, :n] = fill
    return k, v, table


def run_all(pkg, q, w, lens, window, T, kw):
    L = torch.tensor(lens, dtype=torch.int32)
    outs = []
    for fill in (float("nan"), float("inf"), -0.5):
        k, v, table = poisoned(w, lens, window, T, fill)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = pkg.decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), table.to(DEV), L.to(DEV),
                              w.scale, window=window, max_seq_len=max(lens), err_flag=err, **kw)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    if T > 1:
        ref = oracle.decode_attn_multi(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window)
    else:
        ref = oracle.decode_attn(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, window)
    return outs[0], ref


@pytest.mark.parametrize("D,Hq,Hkv,PS,lens,T,window,dtype,chunk,schedule,variant", [
    (128, 32, 8, 16, [3000, 40, 0, 700], 1, 0, torch.float16, 0, AUTO, V_AUTO),
    (128, 32, 8, 16, [3000, 40, 0, 700], 1, 0, torch.float16, 256, GRID, V_AUTO),
    (128, 32, 8, 16, [1500, 40, 0, 700], 1, 0, torch.float16, 512, CLUSTER, V_AUTO),
    (128, 16, 4, 16, [3000], 1, 0, torch.float16, 192, CLUSTER, V_AUTO),  # 16-CTA clusters
    (128, 32, 8, 16, [3000, 40, 0, 700], 1, 0, torch.float16, 0, AUTO, V_SIMT),
    (128, 32, 8, 16, [200, 17, 0, 256], 1, 0, torch.float16, 0, AUTO, V_AUTO),   # single pass
    (64, 16, 4, 16, [5000, 100, 1, 333], 1, 0, torch.float16, 512, GRID, V_AUTO),
    (64, 16, 4, 16, [2000, 100, 1, 333], 1, 0, torch.bfloat16, 512, CLUSTER, V_AUTO),
    (256, 16, 4, 16, [2500, 65, 0, 900], 1, 0, torch.bfloat16, 512, GRID, V_AUTO),
    (128, 16, 4, 32, [2600, 90, 3], 2, 0, torch.float16, 256, GRID, V_AUTO),     # T = 2
    (128, 8, 8, 8, [1900, 20, 700], 1, 0, torch.float16, 384, AUTO, V_AUTO),     # 8-token pages
    (128, 32, 8, 16, [3000, 40, 0, 1707], 1, 700, torch.float16, 0, AUTO, V_AUTO),  # window
    (128, 32, 8, 16, [3000, 40, 0, 1707], 1, 700, torch.float16, 0, AUTO, V_SIMT),
    (128, 16, 4, 32, [2600, 90, 3, 1001], 2, 500, torch.float16, 0, GRID, V_AUTO),
    (64, 16, 4, 32, [3000], 1, 0, torch.bfloat16, 256, CLUSTER, V_AUTO),  # 12-CTA clusters
    (128, 32, 8, 16, [3000, 40, 0, 1707], 1, 700, torch.float16, 0, CLUSTER, V_AUTO),
])
def test_unattended_positions_leave_no_trace(pkg, D, Hq, Hkv, PS, lens, T, window, dtype, chunk,
                                             schedule, variant):
    w = workloads.make_custom("poison", batch=len(lens), num_q_heads=Hq, num_kv_heads=Hkv,
                              head_dim=D, page_size=PS, seq_lens=[max(L, 1) for L in lens],
                              seed=900 + D + PS + window, decoy_pages=2, dtype=dtype)
    g = torch.Generator().manual_seed(901 + D)
    q = torch.randn(len(lens), T, Hq, D, generator=g).to(dtype) if T > 1 else w.q
    out, ref = run_all(pkg, q, w, lens, window, T,
                       dict(schedule=schedule, variant=variant, force_chunk=chunk))
    check(out, ref, dtype)


def test_unattended_positions_many_waves(pkg):
    """A step of several waves: 300 sequences of 1..500 positions, on the
    planner's pick (the shallow ring at D = 128)."""
    lens = [int(x) for x in torch.randint(1, 501, (300,), generator=torch.Generator().manual_seed(7))]
    lens[5] = 0
    w = workloads.make_custom("poison_waves", batch=len(lens), num_q_heads=32, num_kv_heads=8,
                              head_dim=128, page_size=16, seq_lens=[max(L, 1) for L in lens],
                              seed=907)
    params = pkg.make_params(w.q.to(DEV), w.k_pages.to(DEV), w.page_table.to(DEV), w.scale, 0,
                             max(lens), 0, 0, 0, AUTO)
    plan = pkg.decode_attn_make_plan(params,
                                     torch.cuda.get_device_properties(DEV).multi_processor_count)
    assert plan.head_fastest == 1 and plan.ring_stages == 2, plan.as_dict()
    out, ref = run_all(pkg, w.q, w, lens, 0, 1, {})
    check(out, ref, torch.float16)
