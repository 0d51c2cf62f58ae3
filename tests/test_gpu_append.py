"""GPU parity of the paged K/V append (the step before attention) and of the
fused append + attention launch, against the f64 oracle's append and
attention on the same seeded inputs.  The append is a copy, so the pools are
compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS, ROW_REL = 5e-4, 2e-3, 1e-3
DEV = "cuda:0"
VARIANTS = pytest.mark.parametrize("variant", [1, 2], ids=["simt", "mma"])


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


def pool(seed, B, Hq, Hkv, D, PS, lens, spare=1):
    """A pool whose tables leave `spare` free slots after each sequence for
    the new rows (pages allocated up to len + spare)."""
    return workloads.make_custom("a", batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                 page_size=PS, seq_lens=[L + spare for L in lens], seed=seed,
                                 decoy_pages=3)


def new_rows(seed, B, Hkv, D):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(B, Hkv, D, generator=g).half()
    v = torch.randn(B, Hkv, D, generator=g).half()
    return k, v


def u16(t):
    return torch.from_numpy(np.ascontiguousarray(t).view(np.int16)).view(torch.float16)


def check_parity(out, ref):
    g = out.float().cpu().numpy().astype(np.float64).reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    rn = np.linalg.norm(r, axis=1)
    rrel = (np.linalg.norm(g - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    assert rel <= REL_L2 and np.abs(g - r).max() <= MAX_ABS and rrel <= ROW_REL, (rel, rrel)


@pytest.mark.parametrize("PS,D", [(16, 64), (64, 128), (8, 256), (32, 128)])
def test_kv_append_is_bit_exact(pkg, PS, D):
    lens = [0, 5, 31, 64, 100]
    w = pool(40, len(lens), 8, 4, D, PS, lens)
    kn, vn = new_rows(41, len(lens), 4, D)
    pos = torch.tensor([0, 5, 31, -1, 100], dtype=torch.int32)
    ref_k, ref_v, err = oracle.kv_append(kn, vn, pos, w.page_table, w.k_pages, w.v_pages)
    assert err.tolist() == [0] * len(lens)
    kp, vp = w.k_pages.to(DEV), w.v_pages.to(DEV)
    errf = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkg.decode_kv_append(kn.to(DEV), vn.to(DEV), pos.to(DEV), kp, vp, w.page_table.to(DEV),
                         err_flag=errf)
    torch.cuda.synchronize()
    assert int(errf.item()) == 0
    assert torch.equal(kp.cpu(), u16(ref_k).view(kp.shape))
    assert torch.equal(vp.cpu(), u16(ref_v).view(vp.shape))


def test_kv_append_rejects_bad_positions_and_pages(pkg):
    lens = [10, 10, 10]
    w = pool(42, 3, 4, 2, 64, 16, lens)
    kn, vn = new_rows(43, 3, 2, 64)
    table = w.page_table.clone()
    table[1, 0] = w.k_pages.shape[0] + 1
    cap = table.shape[1] * 16
    pos = torch.tensor([cap, 3, 4], dtype=torch.int32)
    kp, vp = w.k_pages.to(DEV), w.v_pages.to(DEV)
    errf = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkg.decode_kv_append(kn.to(DEV), vn.to(DEV), pos.to(DEV), kp, vp, table.to(DEV),
                         err_flag=errf)
    torch.cuda.synchronize()
    assert int(errf.item()) == pkg.DEV_BAD_LEN | pkg.DEV_BAD_PAGE
    ref_k, ref_v, err = oracle.kv_append(kn, vn, pos, table, w.k_pages, w.v_pages)
    assert err.tolist() == [1, 1, 0]
    assert torch.equal(kp.cpu(), u16(ref_k).view(kp.shape))


@VARIANTS
@pytest.mark.parametrize("case", ["llama", "mixed", "window"])
def test_fused_append_attention(pkg, variant, case):
    if case == "llama":
        lens, Hq, Hkv, D, PS, window = [3059], 32, 8, 128, 16, 0
    elif case == "mixed":
        lens, Hq, Hkv, D, PS, window = [0, 1, 255, 700, 4000], 16, 2, 64, 32, 0
    else:
        lens, Hq, Hkv, D, PS, window = [2000, 90, 513], 16, 4, 128, 64, 300
    B = len(lens)
    w = pool(44, B, Hq, Hkv, D, PS, lens)
    kn, vn = new_rows(45, B, Hkv, D)
    L_after = torch.tensor([L + 1 if L > 0 else 0 for L in lens], dtype=torch.int32)
    pos = L_after - 1  # seq_len 0 -> -1 -> no row
    ref_k, ref_v, _ = oracle.kv_append(kn, vn, pos, w.page_table, w.k_pages, w.v_pages)
    ref_out = oracle.decode_attn(w.q, ref_k, ref_v, w.page_table, L_after, w.scale, window)
    kp, vp = w.k_pages.to(DEV), w.v_pages.to(DEV)
    errf = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.decode_attn_append(w.q.to(DEV), kn.to(DEV), vn.to(DEV), kp, vp,
                                 w.page_table.to(DEV), L_after.to(DEV), w.scale, window=window,
                                 max_seq_len=int(L_after.max()), err_flag=errf,
                                 variant=variant)
    torch.cuda.synchronize()
    assert int(errf.item()) == 0
    assert torch.equal(kp.cpu(), u16(ref_k).view(kp.shape))
    assert torch.equal(vp.cpu(), u16(ref_v).view(vp.shape))
    check_parity(out, ref_out)
    # the same bits as the two-launch path (append kernel, then decode_attn)
    kp2, vp2 = w.k_pages.to(DEV), w.v_pages.to(DEV)
    pkg.decode_kv_append(kn.to(DEV), vn.to(DEV), pos.to(DEV), kp2, vp2, w.page_table.to(DEV))
    out2 = pkg.decode_attn(w.q.to(DEV), kp2, vp2, w.page_table.to(DEV), L_after.to(DEV),
                           w.scale, window=window, max_seq_len=int(L_after.max()),
                           variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_decode_loop(pkg):
    """Four decode steps on a growing cache: each step appends its rows with
    the fused launch and attends; the oracle replays the same steps."""
    lens = [100, 37, 256]
    B, Hq, Hkv, D, PS = 3, 16, 4, 128, 16
    w = pool(46, B, Hq, Hkv, D, PS, lens, spare=8)
    kp, vp, table = w.k_pages.to(DEV), w.v_pages.to(DEV), w.page_table.to(DEV)
    ok, ov = w.k_pages.clone(), w.v_pages.clone()
    L = torch.tensor(lens, dtype=torch.int32)
    g = torch.Generator().manual_seed(47)
    for step in range(4):
        q = torch.randn(B, Hq, D, generator=g).half()
        kn, vn = new_rows(48 + step, B, Hkv, D)
        L = L + 1
        out = pkg.decode_attn_append(q.to(DEV), kn.to(DEV), vn.to(DEV), kp, vp, table,
                                     L.to(DEV), w.scale, max_seq_len=int(L.max()))
        torch.cuda.synchronize()
        ok_np, ov_np, _ = oracle.kv_append(kn, vn, L - 1, w.page_table, ok, ov)
        ok, ov = u16(ok_np).view(ok.shape), u16(ov_np).view(ov.shape)
        check_parity(out, oracle.decode_attn(q, ok, ov, w.page_table, L, w.scale, 0))
    assert torch.equal(kp.cpu(), ok) and torch.equal(vp.cpu(), ov)
