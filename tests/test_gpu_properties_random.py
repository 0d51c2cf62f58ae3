"""Seeded random configurations from the wide space of test_gpu_random
(draw_wide), checked against properties that fix the result bit for bit,
so no oracle is needed:

- the same call twice gives the same bits;
- the split kernel followed by the standalone combine gives the fused
  merge's bits (both merge in ascending shard order with one arithmetic);
- the no-allocation entry point gives decode_attn's bits, or refuses a plan
  whose partials exceed its 8 MiB array with DECODE_ATTN_ERR_SCRATCH_LIMIT;
- NaN written into every pool cell that no query attends (the tails of the
  last pages, the decoy pages, positions before a window) changes nothing;
- appending the step's new K/V rows inside the attention launch gives the
  same pools and output as the standalone append followed by attention
  (mlx-runner / llm-web: the K/V scatter that precedes attention)."""
import pytest
import torch

from tests.test_gpu_random import DEV, draw_wide, wide_call, wide_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_gqa_decode_06_gb300 import build
    build.build()
    import paged_gqa_decode_06_gb300 as p
    p.load_library()
    return p


@pytest.mark.parametrize("seed", range(24))
def test_random_entry_point_properties(pkg, seed):
    c = draw_wide(seed)
    T = c["T"]
    # lengths of at least T, so that the T new rows sit inside each sequence
    w, table, L, q, hint, g = wide_inputs(c, seed, min_len=T)
    q, kp, vp = q.to(DEV), w.k_pages.to(DEV), w.v_pages.to(DEV)
    td, Ld = table.to(DEV), L.to(DEV)
    ref = wide_call(pkg, c, q, kp, vp, td, Ld, w.scale, hint)
    if ref is None:
        pytest.skip("cluster schedule refused for this shape")
    assert torch.equal(ref, wide_call(pkg, c, q, kp, vp, td, Ld, w.scale, hint))

    knobs = dict(window=c["window"], max_seq_len=hint, split_min=c["split_min"],
                 force_chunk=c["force_chunk"], schedule=c["schedule"])
    # split, then the standalone combine
    params = pkg.make_params(q, kp, td, w.scale, c["window"], hint, 0, c["split_min"],
                             c["force_chunk"], c["schedule"])
    plan = pkg.decode_attn_make_plan(params,
                                     torch.cuda.get_device_properties(DEV).multi_processor_count)
    out, ws = pkg.decode_attn_split(q, kp, vp, td, Ld, w.scale, **knobs)
    if plan.split:
        out.zero_()
        pkg.decode_attn_combine(params, Ld, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)

    # the no-allocation entry point
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        o2 = pkg.decode_attn_static_scratch(q, kp, vp, td, Ld, w.scale, err_flag=err, **knobs)
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and torch.equal(o2, ref)
    except pkg.DecodeAttnError as e:
        assert e.code == -11, e

    # NaN in every cell no query attends
    PS = c["PS"]
    unattended = torch.ones(kp.shape[0], PS, dtype=torch.bool)
    for b, Lb in enumerate(L.tolist()):
        start = max(0, Lb - T + 1 - c["window"]) if c["window"] > 0 else 0
        if Lb > start:
            pos = torch.arange(start, Lb)
            unattended[table[b, pos // PS].long(), pos % PS] = False
    m = unattended.to(DEV)
    kn, vn = kp.clone(), vp.clone()
    kn[m] = float("nan")
    vn[m] = float("nan")
    assert torch.equal(wide_call(pkg, c, q, kn, vn, td, Ld, w.scale, hint), ref)

    # fused append + attention against the standalone append, then attention
    k_rows = torch.randn(c["B"], T, c["Hkv"], c["D"], generator=g).to(c["dtype"]).to(DEV)
    v_rows = torch.randn(c["B"], T, c["Hkv"], c["D"], generator=g).to(c["dtype"]).to(DEV)
    ka, va, kb, vb = kp.clone(), vp.clone(), kp.clone(), vp.clone()
    err.zero_()
    kr, vr = (k_rows, v_rows) if T > 1 else (k_rows[:, 0], v_rows[:, 0])
    fused = pkg.decode_attn_append(q, kr, vr, ka, va, td, Ld, w.scale, err_flag=err, **knobs)
    for t in range(T):
        pkg.decode_kv_append(k_rows[:, t].contiguous(), v_rows[:, t].contiguous(),
                             (Ld - T + t).contiguous(), kb, vb, td, err_flag=err)
    after = wide_call(pkg, c, q, kb, vb, td, Ld, w.scale, hint)
    assert int(err.item()) == 0
    assert torch.equal(ka, kb) and torch.equal(va, vb)
    assert torch.equal(fused, after)
