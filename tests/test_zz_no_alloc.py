"""decode_attn_static_scratch: the entry point for callers that cannot
allocate device memory (their memory is held by another framework's
allocator, they sit behind an interface that passes only the call's tensors,
or they cannot pay cudaMalloc's implicit synchronisation).  Its shard
partials live in the library's fixed device array instead of a workspace.

Checked through the C ABI against decode_attn with a caller workspace, on two
calls in a row (the second call finds the first call's partials still in the
array), within the parity tolerance the other GPU tests use.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS = 5e-4, 2e-3
DEV = "cuda:0"


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_gqa_decode_06_gb300 import build
    build.build()
    import paged_gqa_decode_06_gb300 as p
    p.load_library()
    return p


def _close(a, b):
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30)
    return rel <= REL_L2 and np.abs(x - y).max() <= MAX_ABS


@pytest.mark.parametrize("name", ["llama", "long_w4096", "batched"])
def test_static_scratch_matches_workspace_path(pkg, name):
    w = workloads.make(name, device=DEV)
    L = w.max_seq_len()
    params = pkg.make_params(w.q, w.k_pages, w.page_table, w.scale, w.window, L)
    assert 0 < pkg.decode_attn_workspace_size(params, 0) <= 8 << 20  # a split plan
    ref = pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                          window=w.window, max_seq_len=L)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for _ in range(2):
        out = torch.empty_like(w.q)
        pkg.decode_attn_static_scratch(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens,
                                       w.scale, window=w.window, out=out, max_seq_len=L,
                                       err_flag=err)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for out in outs:
        assert _close(out, ref)


def test_static_scratch_rejects_plans_above_its_size(pkg):
    # 64 sequences of 8192 tokens in 64-token shards: 128 shards per row,
    # partials of 64*32*128*(128+2)*4 bytes, far above the 8 MiB array
    big = workloads.make_custom("big", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                page_size=16, seq_lens=[8192] * 64, seed=9, device=DEV)
    with pytest.raises(pkg.DecodeAttnError) as e:
        pkg.decode_attn_static_scratch(big.q, big.k_pages, big.v_pages, big.page_table,
                                       big.seq_lens, big.scale, max_seq_len=8192,
                                       force_chunk=64)
    assert e.value.code == -11 and "static scratch" in str(e.value)
