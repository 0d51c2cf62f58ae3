"""Seeded random configurations against the f64 oracle: head dims, group
sizes, query positions, page sizes, batch and length mixes (zeros included),
windows, element formats, variants and schedules drawn together, so the
planner's choices (single pass, split, one wave or several, deep or shallow
ring, workspace or cluster merge) meet the kernels in combinations the fixed cases do not."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
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


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([64, 128, 256]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    T = int(rng.choice([1, 1, 1, 2, 3, 4]))
    G = int(rng.choice([g for g in (1, 2, 4, 8, 16) if T * g <= 16]))
    PS = int(rng.choice([8, 16, 32, 64, 128]))
    lmax = int(rng.choice([100, 300, 600, 3000, 9000]))
    B = int(rng.integers(1, 41))
    while B > 1 and B * Hkv * G * lmax * D > 3e8:  # keeps the oracle to seconds
        B //= 2
    lens = rng.integers(0, lmax + 1, B)
    lens[rng.random(B) < 0.1] = 0
    window = int(rng.integers(1, lmax + 1)) if rng.random() < 0.3 else 0
    dtype = torch.bfloat16 if rng.random() < 0.3 else torch.float16
    variant = 1 if (T == 1 and G <= 8 and dtype == torch.float16 and rng.random() < 0.2) else 2
    schedule = 1 if (variant == 2 and rng.random() < 0.15) else 0  # the workspace merge
    split_min = int(rng.choice([0, 0, 0, 1, 100000]))
    force_chunk = int(rng.choice([0, 0, 0, 0, 64, 192, 1024]))
    return dict(D=D, Hkv=Hkv, G=G, T=T, PS=PS, B=B, lens=lens.tolist(), window=window,
                dtype=dtype, variant=variant, schedule=schedule, split_min=split_min,
                force_chunk=force_chunk, lmax=lmax)


# seeds 0..39, plus three drawn from a wider sweep that ask for a single
# pass over more positions than one shard holds (pages of 8, split_min
# 100000, contexts near 9000)
@pytest.mark.parametrize("seed", list(range(40)) + [98, 204, 419])
def test_random_configuration_matches_oracle(pkg, seed):
    c = draw(seed)
    Hq = c["Hkv"] * c["G"]
    w = workloads.make_custom("r", batch=c["B"], num_q_heads=Hq, num_kv_heads=c["Hkv"],
                              head_dim=c["D"], page_size=c["PS"],
                              seq_lens=[max(L, 1) for L in c["lens"]], seed=2000 + seed,
                              decoy_pages=2, dtype=c["dtype"])
    L = torch.tensor(c["lens"], dtype=torch.int32)
    g = torch.Generator().manual_seed(3000 + seed)
    if c["T"] > 1:
        q = torch.randn(c["B"], c["T"], Hq, c["D"], generator=g).to(c["dtype"])
        ref = oracle.decode_attn_multi(q, w.k_pages, w.v_pages, w.page_table, L, w.scale,
                                       c["window"])
    else:
        q = w.q
        ref = oracle.decode_attn(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, c["window"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.decode_attn(q.to(DEV), w.k_pages.to(DEV), w.v_pages.to(DEV),
                          w.page_table.to(DEV), L.to(DEV), w.scale, window=c["window"],
                          max_seq_len=max(1, c["lmax"]), err_flag=err, variant=c["variant"],
                          split_min=c["split_min"], force_chunk=c["force_chunk"],
                          schedule=c["schedule"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0, c
    rel_t, mab_t, row_t = TOL[c["dtype"]]
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, c["D"])
    r = ref.reshape(-1, c["D"])
    rn = np.linalg.norm(r, axis=1)
    assert np.all(got[rn == 0] == 0), c
    rel = np.linalg.norm(got - r) / max(np.linalg.norm(r), 1e-30)
    rrel = (np.linalg.norm(got - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert rel <= rel_t and np.abs(got - r).max() <= mab_t and rrel <= row_t, (c, rel, rrel)


def draw_many_short(seed):
    """Several waves of short one-shard CTAs: the shallow ring's plans."""
    rng = np.random.default_rng(5000 + seed)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([2, 4, 8]))
    T = int(rng.choice([1, 1, 2]))
    G = int(rng.choice([g for g in (1, 2, 4, 8) if T * g <= 8]))
    lmax = int(rng.choice([256, 512]))
    B = int(rng.integers(200, 401))
    lens = rng.integers(0, lmax + 1, B)
    window = int(rng.integers(1, lmax + 1)) if rng.random() < 0.3 else 0
    dtype = torch.bfloat16 if rng.random() < 0.3 else torch.float16
    return dict(D=D, Hkv=Hkv, G=G, T=T, PS=int(rng.choice([8, 16, 32])), B=B,
                lens=lens.tolist(), window=window, dtype=dtype, variant=2, schedule=0,
                split_min=0, force_chunk=0, lmax=lmax)


@pytest.mark.parametrize("seed", range(8))
def test_random_many_short_matches_oracle(pkg, seed):
    c = draw_many_short(seed)
    Hq = c["Hkv"] * c["G"]
    params = pkg.DecodeAttnParams(
        batch=c["B"], num_q_heads=Hq, num_kv_heads=c["Hkv"], head_dim=c["D"],
        page_size=c["PS"], max_pages_per_seq=(c["lmax"] + c["PS"] - 1) // c["PS"],
        num_pages=10, max_seq_len=c["lmax"], scale=0.1, window=c["window"], variant=2,
        split_min=0, force_chunk=0, num_queries=c["T"],
        dtype=1 if c["dtype"] == torch.bfloat16 else 0, schedule=0)
    plan = pkg.decode_attn_make_plan(params,
                                     torch.cuda.get_device_properties(DEV).multi_processor_count)
    assert plan.ring_stages in (2, 4), plan.as_dict()
    _check(pkg, c, seed)


def _check(pkg, c, seed):
    Hq = c["Hkv"] * c["G"]
    w = workloads.make_custom("s", batch=c["B"], num_q_heads=Hq, num_kv_heads=c["Hkv"],
                              head_dim=c["D"], page_size=c["PS"],
                              seq_lens=[max(L, 1) for L in c["lens"]], seed=6000 + seed,
                              decoy_pages=2, dtype=c["dtype"])
    L = torch.tensor(c["lens"], dtype=torch.int32)
    g = torch.Generator().manual_seed(7000 + seed)
    if c["T"] > 1:
        q = torch.randn(c["B"], c["T"], Hq, c["D"], generator=g).to(c["dtype"])
        ref = oracle.decode_attn_multi(q, w.k_pages, w.v_pages, w.page_table, L, w.scale,
                                       c["window"])
    else:
        q = w.q
        ref = oracle.decode_attn(q, w.k_pages, w.v_pages, w.page_table, L, w.scale, c["window"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.decode_attn(q.to(DEV), w.k_pages.to(DEV), w.v_pages.to(DEV),
                          w.page_table.to(DEV), L.to(DEV), w.scale, window=c["window"],
                          max_seq_len=c["lmax"], err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, c
    rel_t, mab_t, row_t = TOL[c["dtype"]]
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, c["D"])
    r = ref.reshape(-1, c["D"])
    rn = np.linalg.norm(r, axis=1)
    assert np.all(got[rn == 0] == 0), c
    rel = np.linalg.norm(got - r) / max(np.linalg.norm(r), 1e-30)
    rrel = (np.linalg.norm(got - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert rel <= rel_t and np.abs(got - r).max() <= mab_t and rrel <= row_t, (c, rel, rrel)


def draw_wide(seed):
    """A wider space: page sizes up to 256, contexts up to 70000, every
    schedule, forced chunks and thresholds, windows of 1 and beyond the
    length, a length bound above the longest sequence."""
    rng = np.random.default_rng(77000 + seed)
    D = int(rng.choice([64, 128, 256]))
    Hkv = int(rng.choice([1, 2, 4, 8, 16]))
    T = int(rng.choice([1, 1, 1, 2, 3, 4]))
    G = int(rng.choice([g for g in (1, 2, 4, 8, 16) if T * g <= 16]))
    PS = int(rng.choice([8, 16, 32, 64, 128, 256]))
    lmax = int(rng.choice([1, 50, 256, 257, 1000, 5000, 20000, 70000]))
    B = int(rng.integers(1, 65))
    while B > 1 and B * Hkv * G * T * lmax * D > 3e8:  # keeps the oracle to seconds
        B //= 2
    if B * Hkv * G * T * lmax * D > 3e8:
        Hkv = 1
    lens = rng.integers(0, lmax + 1, B)
    lens[rng.random(B) < 0.1] = 0
    lens[rng.random(B) < 0.2] = lmax
    r = rng.random()
    window = 0 if r < 0.6 else (1 if r < 0.65 else int(rng.integers(1, 2 * lmax + 2)))
    dtype = torch.bfloat16 if rng.random() < 0.3 else torch.float16
    schedule = int(rng.choice([0, 0, 1, 2]))
    split_min = int(rng.choice([0, 0, 1, 64, 100000]))
    force_chunk = int(rng.choice([0, 0, 0, 64, 128, 640, 4096]))
    hint = lmax if rng.random() < 0.8 else lmax + int(rng.integers(1, 5000))
    return dict(D=D, Hkv=Hkv, G=G, T=T, PS=PS, B=B, lens=lens.tolist(), window=window,
                dtype=dtype, schedule=schedule, split_min=split_min, force_chunk=force_chunk,
                lmax=lmax, hint=hint)


def wide_inputs(c, seed, min_len=0):
    """Pools, a page table padded to the length bound, lengths and queries."""
    Hq = c["Hkv"] * c["G"]
    lens = [max(L, min_len) for L in c["lens"]]
    w = workloads.make_custom("w", batch=c["B"], num_q_heads=Hq, num_kv_heads=c["Hkv"],
                              head_dim=c["D"], page_size=c["PS"],
                              seq_lens=[max(L, 1) for L in lens], seed=8000 + seed,
                              decoy_pages=2, dtype=c["dtype"])
    hint = max(c["hint"], max(lens))
    table = w.page_table
    need = (hint + c["PS"] - 1) // c["PS"]
    if table.shape[1] < need:
        pad = torch.full((table.shape[0], need - table.shape[1]), -1, dtype=torch.int32)
        table = torch.cat([table, pad], 1).contiguous()
    g = torch.Generator().manual_seed(9000 + seed)
    shape = (c["B"], c["T"], Hq, c["D"]) if c["T"] > 1 else (c["B"], Hq, c["D"])
    q = torch.randn(*shape, generator=g).to(c["dtype"])
    return w, table, torch.tensor(lens, dtype=torch.int32), q, hint, g


def wide_call(pkg, c, q, k, v, table, L, scale, hint, **kw):
    """decode_attn with the draw's knobs; None when the cluster schedule is
    refused for the shape (DECODE_ATTN_ERR_VARIANT, documented)."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        out = pkg.decode_attn(q, k, v, table, L, scale, window=c["window"], max_seq_len=hint,
                              err_flag=err, split_min=c["split_min"],
                              force_chunk=c["force_chunk"], schedule=c["schedule"], **kw)
    except pkg.DecodeAttnError as e:
        if e.code == -10 and c["schedule"] == 2:
            return None
        raise
    torch.cuda.synchronize()
    assert int(err.item()) == 0, c
    return out


@pytest.mark.parametrize("seed", range(24))
def test_wide_configuration_matches_oracle(pkg, seed):
    c = draw_wide(seed)
    w, table, L, q, hint, _ = wide_inputs(c, seed)
    out = wide_call(pkg, c, q.to(DEV), w.k_pages.to(DEV), w.v_pages.to(DEV), table.to(DEV),
                    L.to(DEV), w.scale, hint)
    if out is None:
        pytest.skip("cluster schedule refused for this shape")
    if c["T"] > 1:
        ref = oracle.decode_attn_multi(q, w.k_pages, w.v_pages, table, L, w.scale, c["window"])
    else:
        ref = oracle.decode_attn(q, w.k_pages, w.v_pages, table, L, w.scale, c["window"])
    rel_t, mab_t, row_t = TOL[c["dtype"]]
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, c["D"])
    r = ref.reshape(-1, c["D"])
    rn = np.linalg.norm(r, axis=1)
    assert np.all(got[rn == 0] == 0), c
    rel = np.linalg.norm(got - r) / max(np.linalg.norm(r), 1e-30)
    rrel = (np.linalg.norm(got - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert rel <= rel_t and np.abs(got - r).max() <= mab_t and rrel <= row_t, (c, rel, rrel)
