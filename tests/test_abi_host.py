"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/*.h declares, rejects bad arguments before touching
the device, and the planner's choices obey their contract."""
import ctypes
import glob
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    from paged_gqa_decode_06_gb300 import build
    build.build()
    import paged_gqa_decode_06_gb300 as p
    p.load_library()
    return p


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if not m.group(0).lstrip().startswith(("#", "typedef", "return")):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("decode_attn", "decode_attn_split", "decode_attn_combine", "decode_attn_host",
              "decode_attn_workspace_size", "decode_attn_make_plan", "decode_attn_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(pkg):
    lib = ctypes.CDLL(pkg.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_needs_no_driver_at_load(pkg):
    # cudart is static; the driver is only reached on the first CUDA call
    out = os.popen(f"ldd {pkg.library_path()}").read()
    assert "libcuda.so" not in out
    assert "libtorch" not in out


def params(pkg, **kw):
    base = dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                max_pages_per_seq=192, num_pages=256, max_seq_len=3060, scale=0.088,
                window=0, variant=0, split_min=0, force_chunk=0, num_queries=1, dtype=0,
                schedule=0)
    base.update(kw)
    return pkg.DecodeAttnParams(**base)


def test_strerror(pkg):
    assert pkg.decode_attn_strerror(0) == "ok"
    assert "head_dim" in pkg.decode_attn_strerror(-3)
    assert pkg.decode_attn_strerror(-999) == "unknown status"


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, -3), ("page_size", 24, -4), ("page_size", 4, -4), ("page_size", 512, -4),
    ("num_q_heads", 30, -2), ("num_kv_heads", 0, -2), ("batch", -1, -2),
    ("max_pages_per_seq", 0, -2), ("num_pages", 0, -2), ("scale", float("nan"), -2),
    ("num_q_heads", 8 * 32, -5),
])
def test_bad_params_rejected_before_launch(pkg, field, value, code):
    p = params(pkg, **{field: value})
    plan = pkg.DecodeAttnPlan()
    lib = pkg.load_library()
    assert lib.decode_attn_make_plan(ctypes.byref(p), 152, ctypes.byref(plan)) == code
    # the launch entry points return the same code without any CUDA call
    nul = None
    assert lib.decode_attn(ctypes.byref(p), nul, nul, nul, nul, nul, nul, nul, 0, nul,
                           nul) == code


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, -3), ("page_size", 24, -4), ("num_q_heads", 30, -2),
    ("num_q_heads", 8 * 32, -5), ("scale", float("inf"), -2),
])
def test_static_scratch_rejects_bad_params_without_a_device(pkg, field, value, code):
    # the no-allocation entry point checks its arguments with the planner's
    # parameter checks before any CUDA call (no plan at a made-up SM count)
    lib = pkg.load_library()
    f = lib.decode_attn_static_scratch
    f.argtypes = [ctypes.POINTER(pkg.DecodeAttnParams)] + [ctypes.c_void_p] * 8
    f.restype = ctypes.c_int
    p = params(pkg, **{field: value})
    assert f(ctypes.byref(p), *([None] * 8)) == code
    assert f(None, *([None] * 8)) == -1


def test_null_params(pkg):
    lib = pkg.load_library()
    assert lib.decode_attn(None, None, None, None, None, None, None, None, 0, None, None) == -1
    plan = pkg.DecodeAttnPlan()
    assert lib.decode_attn_make_plan(None, 152, ctypes.byref(plan)) == -1


def test_short_context_single_pass(pkg):
    for L in (1, 64, 200, 256):
        plan = pkg.decode_attn_make_plan(params(pkg, max_seq_len=L), 152)
        assert plan.split == 0 and plan.max_shards == 1
        assert plan.chunk_tokens >= L and plan.chunk_tokens % 64 == 0
        assert plan.workspace_bytes == 0


def test_threshold_at_256(pkg):
    # contexts above 256 split (apache/tvm pull request 20426: "> 256")
    plan = pkg.decode_attn_make_plan(params(pkg, max_seq_len=257), 152)
    assert plan.split == 1 and plan.max_shards >= 2
    plan = pkg.decode_attn_make_plan(params(pkg, max_seq_len=300, split_min=512), 152)
    assert plan.split == 0


@pytest.mark.parametrize("page_size,length,shards", [(8, 9000, 2), (8, 8192, 1),
                                                     (16, 40000, 3), (64, 9000, 1)])
def test_single_pass_request_longer_than_one_shard_splits(pkg, page_size, length, shards):
    """A split threshold above the context asks for one shard, but a shard
    holds at most 1024 TMA boxes of min(page, 64) positions: a longer range
    is cut into the fewest shards that fit instead of being refused."""
    p = params(pkg, page_size=page_size, max_pages_per_seq=(length + page_size - 1) // page_size,
               num_pages=4096, max_seq_len=length, split_min=100000)
    plan = pkg.decode_attn_make_plan(p, 152)
    box = min(page_size, 64)
    assert plan.max_shards == shards and plan.split == (shards > 1)
    assert plan.chunk_tokens <= 1024 * box and plan.chunk_tokens % 64 == 0


def test_few_units_take_one_wave(pkg):
    # B=4, Hkv=8, 131072 tokens, D=128: 32 (b, h) units on 152 SMs x 2 CTAs.
    # Fewer units than slots: one wave, shard count from the cost model
    # (stream rate against one merge round trip per 8 shards): 8 shards, 256
    # CTAs (the chunk sweep's best; 1.7 waves and 1.26 waves measured slower)
    p = params(pkg, batch=4, num_q_heads=64, num_kv_heads=8, page_size=64,
               max_pages_per_seq=2048, num_pages=8192, max_seq_len=131072, schedule=1)
    plan = pkg.decode_attn_make_plan(p, 152)
    slots = 152 * plan.ctas_per_sm
    ctas = plan.grid_x * plan.grid_y * plan.grid_z
    assert plan.split == 1
    assert plan.chunk_tokens * plan.max_shards >= 131072
    assert plan.max_shards == 8 and ctas == 256 and ctas <= slots, (ctas, slots)
    assert plan.workspace_bytes >= 64 * 1024 + 4 * 64 * plan.max_shards * (128 + 2) * 4


@pytest.mark.parametrize("batch,max_len,shards", [
    (1, 131072, 32),   # one long sequence: 256 CTAs (89.1 us; 24 shards 92.0, 38 shards 94.3)
    (1, 16384, 24),    # 192 CTAs (24.95 us; 16 shards 24.5, 32 shards 25.2)
    (2, 65536, 16),    # 256 CTAs (87.5 us; 19 shards 90.0, 32 shards 91.8)
    (4, 32768, 8),     # 256 CTAs (85.9 us; 16 shards 89.7)
])
def test_one_wave_cost_model_picks(pkg, batch, max_len, shards):
    # the picks the model makes on the chunk sweep's shapes (64/8 heads,
    # D=128, page 64), each the measured best or within 2 % of it; grids stay
    # near 0.85 of the CTA slots
    p = params(pkg, batch=batch, num_q_heads=64, num_kv_heads=8, page_size=64,
               max_pages_per_seq=max_len // 64, num_pages=batch * max_len // 64,
               max_seq_len=max_len, schedule=1)
    plan = pkg.decode_attn_make_plan(p, 152)
    assert plan.max_shards == shards
    assert plan.grid_x * plan.grid_y * plan.grid_z <= 152 * plan.ctas_per_sm
    assert plan.head_fastest == 0


def test_one_wave_plan_never_exceeds_the_slots(pkg):
    for B in (1, 2, 3, 5, 7, 9, 16, 37):
        for L in (300, 1000, 3060, 20000, 131072):
            p = params(pkg, batch=B, max_pages_per_seq=(L + 15) // 16, num_pages=10,
                       max_seq_len=L, schedule=1)
            plan = pkg.decode_attn_make_plan(p, 152)
            ctas = plan.grid_x * plan.grid_y * plan.grid_z
            if B * 8 < 152 * 2 and L > 256:
                # unless the split's minimum of two shards, or the shard's page
                # ids (1024 per shard, page 16), force more shards
                assert plan.max_shards >= 2
                assert ctas <= 152 * plan.ctas_per_sm or \
                    plan.max_shards == max(2, math.ceil(L / (1024 * 16))), (B, L, ctas)
                assert plan.chunk_tokens >= 128 or plan.max_shards == 1


def test_mixed_lengths_get_bounded_chunks(pkg):
    # B=64 lengths up to 8192: chunks of at most 2048 tokens keep the pieces
    # of short and long sequences balanced
    p = params(pkg, batch=64, max_pages_per_seq=512, num_pages=18000, max_seq_len=8192,
               schedule=1)
    plan = pkg.decode_attn_make_plan(p, 152)
    assert plan.chunk_tokens <= 2048 and plan.max_shards >= 4


def test_small_work_uses_one_wave(pkg):
    for p in (params(pkg),  # Llama-3.1-8B shape, 3060 tokens
              params(pkg, batch=4, num_q_heads=64, page_size=64, max_pages_per_seq=2048,
                     num_pages=8192, max_seq_len=131072, window=4096)):
        plan = pkg.decode_attn_make_plan(p, 152)
        ctas = plan.grid_x * plan.grid_y * plan.grid_z
        assert ctas <= 152 * plan.ctas_per_sm and plan.chunk_tokens >= 128


def test_window_plan_bounds_grid(pkg):
    p = params(pkg, batch=4, num_q_heads=64, num_kv_heads=8, page_size=64,
               max_pages_per_seq=2048, num_pages=8192, max_seq_len=131072, window=4096)
    plan = pkg.decode_attn_make_plan(p, 152)
    # the grid covers the window plus the tile-alignment slack, not the context
    assert plan.chunk_tokens * plan.max_shards >= 4096 + 63
    assert plan.chunk_tokens * (plan.max_shards - 1) < 4096 + 63


def test_force_chunk(pkg):
    plan = pkg.decode_attn_make_plan(params(pkg, force_chunk=100), 152)
    assert plan.chunk_tokens == 128
    assert plan.max_shards == math.ceil(3060 / 128)
    with pytest.raises(pkg.DecodeAttnError):
        pkg.decode_attn_make_plan(params(pkg, force_chunk=1 << 20), 152)


def test_plan_is_a_pure_function(pkg):
    a = pkg.decode_attn_make_plan(params(pkg), 152).as_dict()
    b = pkg.decode_attn_make_plan(params(pkg), 152).as_dict()
    assert a == b
    c = pkg.decode_attn_make_plan(params(pkg), 76).as_dict()
    assert c["chunk_tokens"] >= a["chunk_tokens"]


@pytest.mark.parametrize("max_len", [257, 1000, 3060, 8192, 65536, 131072])
@pytest.mark.parametrize("units", [(1, 8), (64, 8), (4, 8), (1, 1)])
def test_plan_covers_every_length(pkg, max_len, units):
    B, Hkv = units
    PS = 16
    p = params(pkg, batch=B, num_kv_heads=Hkv, num_q_heads=Hkv * 4,
               max_pages_per_seq=(max_len + PS - 1) // PS, num_pages=10, max_seq_len=max_len,
               schedule=1)
    plan = pkg.decode_attn_make_plan(p, 152)
    assert plan.chunk_tokens % 64 == 0
    assert plan.chunk_tokens * plan.max_shards >= max_len
    assert plan.chunk_tokens <= 1024 * min(PS, 64)   # page ids of one shard fit in smem
    if plan.head_fastest:
        assert plan.grid_x == Hkv and plan.grid_y == plan.max_shards
    else:
        assert plan.grid_x == plan.max_shards and plan.grid_y == Hkv
    assert plan.grid_z == B
    slots = 152 * plan.ctas_per_sm
    assert bool(plan.head_fastest) == (B * Hkv * plan.max_shards > slots)


def declared_arity():
    out = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(([^)]*)\)\s*;",
                             text, flags=re.M):
            args = m.group(2).strip()
            out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argtypes_match_header(pkg):
    lib = pkg.load_library()
    arity = declared_arity()
    assert arity
    for name, n in arity.items():
        f = getattr(lib, name)
        if f.argtypes is not None:
            assert len(f.argtypes) == n, (name, len(f.argtypes), n)


def test_variant_selection(pkg):
    # explicit CUDA-core variant serves groups up to 8 heads
    with pytest.raises(pkg.DecodeAttnError) as e:
        pkg.decode_attn_make_plan(params(pkg, num_q_heads=64, num_kv_heads=4, variant=1), 152)
    assert e.value.code == -10
    # tensor-core variant: one n8 tile up to 8 heads, two up to 16
    plan = pkg.decode_attn_make_plan(params(pkg, num_q_heads=64, num_kv_heads=4, variant=2), 152)
    assert plan.variant == 2 and plan.group_pad == 16
    plan = pkg.decode_attn_make_plan(params(pkg, num_q_heads=12, num_kv_heads=4, variant=2), 152)
    assert plan.group_pad == 8
    plan = pkg.decode_attn_make_plan(params(pkg, num_q_heads=12, num_kv_heads=4, variant=1), 152)
    assert plan.variant == 1 and plan.group_pad == 4
    with pytest.raises(pkg.DecodeAttnError):
        pkg.decode_attn_make_plan(params(pkg, variant=7), 152)
    # automatic choice is a pure function of the shape
    a = pkg.decode_attn_make_plan(params(pkg), 152).variant
    assert a in (1, 2) and a == pkg.decode_attn_make_plan(params(pkg), 152).variant


def test_multi_query_plans(pkg):
    # T query positions per sequence: T * G rows per KV head on the mma side
    plan = pkg.decode_attn_make_plan(params(pkg, num_queries=2), 152)  # G=4 -> 8 rows
    assert plan.variant == 2 and plan.group_pad == 8
    plan = pkg.decode_attn_make_plan(params(pkg, num_queries=4), 152)  # 16 rows
    assert plan.group_pad == 16
    for bad in (dict(num_queries=5), dict(num_queries=2, variant=1)):
        with pytest.raises(pkg.DecodeAttnError) as e:
            pkg.decode_attn_make_plan(params(pkg, **bad), 152)
        assert e.value.code == -10
    # the window of the first query starts T - 1 positions earlier
    p = params(pkg, batch=1, max_pages_per_seq=2048, num_pages=4096, max_seq_len=30000,
               window=1000, num_queries=4)
    plan = pkg.decode_attn_make_plan(p, 152)
    assert plan.chunk_tokens * plan.max_shards >= 1000 + 3 + 63
    one = pkg.decode_attn_make_plan(params(pkg, num_queries=1), 152)
    four = pkg.decode_attn_make_plan(params(pkg, num_queries=4), 152)
    assert four.workspace_bytes - 65536 >= 4 * (one.workspace_bytes - 65536) - 4096


def test_bf16_plans(pkg):
    plan = pkg.decode_attn_make_plan(params(pkg, dtype=1), 152)
    assert plan.variant == 2
    for bad in (dict(dtype=1, variant=1), dict(dtype=2)):
        with pytest.raises(pkg.DecodeAttnError):
            pkg.decode_attn_make_plan(params(pkg, **bad), 152)


@pytest.mark.parametrize("D,Hq,Hkv,stages", [(128, 32, 8, 2), (64, 32, 8, 4), (64, 64, 4, 4),
                                             (128, 64, 4, None), (256, 16, 4, None)])
def test_shallow_ring_for_many_short_shards(pkg, D, Hq, Hkv, stages):
    # a thousand sequences of up to 512 tokens: several waves of one-shard
    # CTAs take the 2-stage (4 at D=64) ring and 3 CTAs per SM, except where
    # three CTAs per SM do not fit (D=256; D=128 with 16 query rows)
    p = params(pkg, batch=1000, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
               max_pages_per_seq=32, num_pages=40000, max_seq_len=512, schedule=1)
    plan = pkg.decode_attn_make_plan(p, 152)
    assert plan.chunk_tokens <= 512
    if stages is None:
        assert plan.ring_stages == (6 if D == 64 else 3)
    else:
        assert plan.ring_stages == stages and plan.ctas_per_sm == 3


def test_long_shards_keep_the_deep_ring(pkg):
    for p in (params(pkg),  # Llama-3.1-8B shape: one wave
              params(pkg, batch=64, max_pages_per_seq=512, num_pages=18000, max_seq_len=8192,
                     schedule=1),  # batched: 2048-token shards
              params(pkg, batch=4, num_q_heads=64, page_size=64, max_pages_per_seq=2048,
                     num_pages=8192, max_seq_len=131072)):
        plan = pkg.decode_attn_make_plan(p, 152)
        assert plan.ring_stages == 3 and plan.ctas_per_sm == 2


def test_environment_sets_the_planner_defaults():
    """DECODE_ATTN_SPLIT_MIN / DECODE_ATTN_FORCE_CHUNK are read once per
    process; a fresh process sees them (the mlx-runner page's
    MLXR_ATTN_SPLIT_MIN plays this role there)."""
    import os
    import subprocess
    import sys
    code = ("import paged_gqa_decode_06_gb300 as p; p.load_library(); "
            "P = p.DecodeAttnParams(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, "
            "page_size=16, max_pages_per_seq=192, num_pages=256, max_seq_len=400, scale=0.1, "
            "window=0, variant=0, split_min=0, force_chunk=0, num_queries=1, dtype=0, "
            "schedule=0); pl = p.decode_attn_make_plan(P, 152); print(pl.split, pl.chunk_tokens)")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

    def plan_with(env):
        e = dict(os.environ, **env)
        r = subprocess.run([sys.executable, "-c", code], cwd=root, env=e, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        return tuple(int(x) for x in r.stdout.split())

    assert plan_with({})[0] == 1                               # 400 > 256: split
    assert plan_with({"DECODE_ATTN_SPLIT_MIN": "512"})[0] == 0  # threshold moved
    assert plan_with({"DECODE_ATTN_FORCE_CHUNK": "64"}) == (1, 64)


def test_cluster_plans(pkg):
    """One-wave tensor-core split plans of 2..8 shards (9..16 on grids of at
    most 64 CTAs) merge inside a thread-block cluster when the grid fills most
    CTA slots or the step is small; the grid schedule and longer shard lists
    merge through the workspace; asking for a cluster where none applies is an
    error."""
    long4 = dict(batch=4, num_q_heads=64, num_kv_heads=8, page_size=64, max_pages_per_seq=2048,
                 num_pages=8192, max_seq_len=131072)
    plan = pkg.decode_attn_make_plan(params(pkg, **long4), 152)
    assert plan.cluster == plan.max_shards == 8 and plan.head_fastest == 0
    plan = pkg.decode_attn_make_plan(params(pkg, **long4, window=4096), 152)
    assert plan.cluster == plan.max_shards
    plan = pkg.decode_attn_make_plan(params(pkg, **long4, schedule=1), 152)
    assert plan.cluster == 0
    # Llama shape: 16 shards, 128 CTAs: too many for clusters above 8, which
    # only small grids (up to 64 CTAs) take; the head_dim-256 shape does
    plan = pkg.decode_attn_make_plan(params(pkg), 152)
    assert plan.max_shards == 16 and plan.cluster == 0
    plan = pkg.decode_attn_make_plan(params(pkg, num_q_heads=16, num_kv_heads=4, head_dim=256),
                                     152)
    assert plan.cluster == plan.max_shards == 16
    with pytest.raises(pkg.DecodeAttnError):                  # 24 shards
        pkg.decode_attn_make_plan(params(pkg, schedule=2, force_chunk=128), 152)
    plan = pkg.decode_attn_make_plan(params(pkg, schedule=2, force_chunk=384), 152)
    assert plan.cluster == plan.max_shards == 8
    plan = pkg.decode_attn_make_plan(params(pkg, schedule=1), 152)
    assert plan.cluster == 0 and plan.max_shards == 16
    # a sparse grid of clusters (128 CTAs, 537 MB) keeps the workspace merge
    plan = pkg.decode_attn_make_plan(
        params(pkg, batch=2, num_q_heads=64, page_size=64, max_pages_per_seq=1024,
               num_pages=2048, max_seq_len=65536, force_chunk=8192), 152)
    assert plan.max_shards == 8 and plan.cluster == 0
