"""GPU parity on the method's closed forms and on extreme inputs.

The decode-attention definition (apache/tvm pull request 20426, sharded-nest
commit: scaled softmax of q.k over the cached keys, output checked against
an f64 reference to f16 rounding) fixes what these inputs must give:

  * q = 0: every score is zero, the softmax is uniform, out = mean of V;
  * all K rows of a KV head equal: the scores of a row are all equal, so
    again out = mean of V, for any q;
  * all V rows of a KV head equal to c: out = c;
  * a peaked softmax: scale * q.k spanning about +-1000, its largest score
    planted in the middle of the context (not on a shard or tile edge), so
    the running maximum jumps by hundreds and the earlier partial sums must
    be rescaled to nothing;
  * |out| in [4, 8): V rows of one sign per dim with magnitudes in [4, 8),
    where half an fp16 ulp (1.95e-3) nearly fills the 2e-3 bar, so only a
    kernel whose fp32 error stays below ~5e-5 passes.

Each input goes through every kernel path the planner has (single pass, the
grid schedule merging through the workspace, the thread-block-cluster merge,
the shallow ring), in fp16 and bf16, and with two query positions per
sequence; the GPU output is compared element by element with the f64 oracle
at the same bars as the other parity suites (bf16: the bars derived from its
rounding floor, widened to half a bf16 ulp where |out| >= 4)."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

DEV = "cuda:0"
BARS = {torch.float16: (5e-4, 2e-3, 1e-3), torch.bfloat16: (3e-3, 1e-2, 6e-3)}
GRID, CLUSTER = 1, 2

# path -> (shape, lengths, call keywords)
PATHS = {
    "single": (dict(batch=2, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16),
               [200, 137], {}),
    "grid": (dict(batch=2, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16),
             [3000, 1777], dict(schedule=GRID)),
    "cluster": (dict(batch=2, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64),
                [4000, 2900], dict(schedule=CLUSTER, force_chunk=640)),
    "shallow": (dict(batch=48, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16),
                None, dict(force_chunk=128)),
}
KINDS = ["q_zero", "equal_k", "const_v", "peaked", "big_out"]


@pytest.fixture(scope="module")
def pkg():
    from paged_gqa_decode_06_gb300 import build
    build.build()
    oracle.build()
    import paged_gqa_decode_06_gb300 as p
    p.load_library()
    return p


def lengths(path):
    shape, lens, _ = PATHS[path]
    if lens is not None:
        return lens
    g = torch.Generator().manual_seed(11)
    return torch.randint(257, 501, (shape["batch"],), generator=g).tolist()


def check_plan(pkg, path, params):
    plan = pkg.decode_attn_make_plan(params, torch.cuda.get_device_properties(0)
                                     .multi_processor_count)
    if path == "single":
        assert plan.split == 0
    elif path == "grid":
        assert plan.split == 1 and plan.cluster == 0
    elif path == "cluster":
        assert plan.split == 1 and plan.cluster >= 2
    else:  # the shallow ring: 2 stages of 64 tokens at D = 128, several waves
        assert plan.split == 1 and plan.ring_stages == 2
    return plan


def off_edge(pos, chunk, L):
    """A position near `pos` that is neither the first nor the last of its
    64-token tile or of its shard."""
    p = min(max(pos, 9), L - 9)
    while p % 64 in (0, 63) or p % chunk in (0, chunk - 1):
        p += 5
    return p


def make_case(pkg, shape, lens, kw, kind, dtype, T=1):
    """Seeded inputs of one case (host tensors): (workload, q, k_pages,
    v_pages, scale)."""
    w = workloads.make_custom(f"inv_{kind}", seq_lens=lens, seed=23, decoy_pages=3,
                              dtype=dtype, **shape)
    B, Hq, D = shape["batch"], shape["num_q_heads"], shape["head_dim"]
    Hkv = shape["num_kv_heads"]
    G = Hq // Hkv
    g = torch.Generator().manual_seed(29)
    q = w.q if T == 1 else torch.randn(B, T, Hq, D, generator=g).to(dtype)
    k, v, scale = w.k_pages.clone(), w.v_pages.clone(), w.scale
    if kind == "q_zero":
        q = torch.zeros_like(q)
    elif kind == "equal_k":
        k[:] = torch.randn(1, 1, Hkv, D, generator=g).to(dtype)
    elif kind == "const_v":
        v[:] = torch.randn(1, 1, Hkv, D, generator=g).to(dtype)
    elif kind == "big_out":
        sign = torch.where(torch.rand(Hkv, D, generator=g) < 0.5, -1.0, 1.0)
        mag = 4.0 + 3.9 * torch.rand(v.shape, generator=g)
        v = (mag * sign).to(dtype)
    elif kind == "peaked":
        # scale * q.k: the planted key gives scale * |q|^2 ~ 10 * 128 ~ 1300,
        # the others N(0, 10^2 * 128), i.e. scores spread over several hundred
        scale = 10.0
        params = pkg.make_params(q, k[:1], w.page_table, scale, 0, max(lens), **kw)
        chunk = pkg.decode_attn_make_plan(params, 152).chunk_tokens
        PS = shape["page_size"]
        for b in range(B):
            pos = off_edge(lens[b] // 2 + 3, chunk, lens[b])
            phys = int(w.page_table[b, pos // PS])
            for h in range(Hkv):
                k[phys, pos % PS, h] = q[b, h * G] if T == 1 else q[b, T - 1, h * G]
    return w, q, k, v, scale


def compare(out, ref, dtype):
    rel_bar, abs_bar, row_bar = BARS[dtype]
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rel = np.linalg.norm(got - r) / max(np.linalg.norm(r), 1e-30)
    rn = np.linalg.norm(r, axis=1)
    row = (np.linalg.norm(got - r, axis=1) / np.where(rn > 0, rn, 1.0)).max()
    tol = np.full(r.shape, abs_bar)
    if dtype == torch.bfloat16:
        # half a bf16 ulp of |out| (8 significand bits), plus 1 %
        mag = np.maximum(np.abs(r), 2.0 ** -126)
        tol = np.maximum(tol, 1.01 * 2.0 ** (np.floor(np.log2(mag)) - 8))
    err = np.abs(got - r)
    worst = float((err / tol).max())
    assert rel <= rel_bar and row <= row_bar and worst <= 1.0, (rel, row, worst, err.max())
    return rel, err.max()


def run(pkg, w, q, k, v, scale, kw):
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    td, ld = w.page_table.to(DEV), w.seq_lens.to(DEV)
    L = int(w.seq_lens.max())
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pkg.decode_attn(qd, kd, vd, td, ld, scale, max_seq_len=L, err_flag=err, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("path", list(PATHS))
def test_closed_forms_and_extremes(pkg, path, kind, dtype):
    shape, _, kw = PATHS[path]
    lens = lengths(path)
    w, q, k, v, scale = make_case(pkg, shape, lens, kw, kind, dtype)
    ref = oracle.decode_attn(q, k, v, w.page_table, w.seq_lens, scale, 0)
    check_plan(pkg, path, pkg.make_params(q, k, w.page_table, scale, 0, max(lens), **kw))
    out = run(pkg, w, q, k, v, scale, kw)
    compare(out, ref, dtype)
    got = out.float().cpu().numpy()
    G = shape["num_q_heads"] // shape["num_kv_heads"]
    if kind == "const_v":  # out = c, to the element format's rounding
        want = np.repeat(v[0, 0].float().numpy(), G, axis=0)[None]
        assert np.abs(got - want).max() <= BARS[dtype][1]
    if kind == "big_out":  # the tolerance edge is really reached
        assert np.abs(ref).min() >= 4.0 and np.abs(ref).max() < 8.0


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["q_zero", "peaked", "big_out"])
@pytest.mark.parametrize("path", ["single", "grid", "cluster"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
def test_extremes_with_two_query_positions(pkg, path, kind, dtype):
    """T = 2 new positions per sequence (causal among themselves) at G = 8:
    16 query rows per KV row read (two n8 tiles of the tensor-core kernel)."""
    base, lens, kw = PATHS["grid" if path == "single" else path]
    shape = dict(base, num_q_heads=8 * base["num_kv_heads"])
    if path == "single":
        lens, kw = [200, 137], {}
    w, q, k, v, scale = make_case(pkg, shape, lens, kw, kind, dtype, T=2)
    ref = oracle.decode_attn_multi(q, k, v, w.page_table, w.seq_lens, scale, 0)
    plan = pkg.decode_attn_make_plan(pkg.make_params(q, k, w.page_table, scale, 0, max(lens),
                                                     **kw),
                                     torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan.group_pad == 16
    if path == "single":
        assert plan.split == 0
    elif path == "cluster":
        assert plan.cluster >= 2
    else:
        assert plan.split == 1 and plan.cluster == 0
    out = run(pkg, w, q, k, v, scale, kw)
    compare(out, ref, dtype)


def test_peaked_inputs_are_peaked(pkg):
    """Host check of the peaked case's inputs: scores spanning several
    hundred, the largest inside a tile, off every edge."""
    shape, lens, kw = PATHS["grid"]
    w, q, k, v, scale = make_case(pkg, shape, lens, kw, "peaked", torch.float16)
    PS, G = shape["page_size"], shape["num_q_heads"] // shape["num_kv_heads"]
    for b in range(shape["batch"]):
        for h in (0, 5):
            L = int(w.seq_lens[b])
            rows = torch.stack([k[int(w.page_table[b, t // PS]), t % PS, h].double()
                                for t in range(L)])
            s = scale * (rows @ q[b, h * G].double())
            top = int(torch.argmax(s))
            assert s.max() > 700 and s.min() < -200 and math.isfinite(float(s.max()))
            assert top % 64 not in (0, 63) and 0 < top < L - 1
            assert (s.max() - s.topk(2).values[1]) > 100  # one key dominates
