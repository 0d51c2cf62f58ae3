"""decode_attn_static_scratch: the entry point for callers that cannot
allocate device memory (their memory is held by another framework's
allocator, they sit behind an interface that passes only the call's tensors,
or they cannot pay cudaMalloc's implicit synchronisation).  Its shard
partials live in the library's fixed device array instead of a workspace.

Checked through the C ABI against decode_attn with a caller workspace, on two
calls in a row (the second call finds the first call's partials still in the
array).  Both entry points make the same plan and launch the same kernel, so
their outputs must agree bit for bit; the output is also compared with the
f64 oracle at the parity tolerance the other GPU tests use.  A call whose
pipeline wait gives up must not spoil the next one: each call clears the
array's shard tickets itself.  This file is collected last so that a run
stopping at the first failure has already run every other test; it also
passes alone in a fresh process."""
import os

import numpy as np
import pytest
import torch

import oracle
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
    oracle.build()
    import paged_gqa_decode_06_gb300 as p
    p.load_library()
    return p


def _assert_close_to_oracle(out, w):
    wc = w.to("cpu")
    ref = oracle.decode_attn(wc.q, wc.k_pages, wc.v_pages, wc.page_table, wc.seq_lens, wc.scale,
                             w.window)
    x = out.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    rel = np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= REL_L2 and np.abs(x - ref).max() <= MAX_ABS, (w.name, rel)


def _static(pkg, w, err):
    out = torch.empty_like(w.q)
    pkg.decode_attn_static_scratch(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens,
                                   w.scale, window=w.window, out=out, max_seq_len=w.max_seq_len(),
                                   err_flag=err)
    return out


@pytest.mark.parametrize("name", ["llama", "long_w4096", "batched"])
def test_static_scratch_matches_workspace_path(pkg, name):
    w = workloads.make(name, device=DEV)
    L = w.max_seq_len()
    params = pkg.make_params(w.q, w.k_pages, w.page_table, w.scale, w.window, L)
    assert 0 < pkg.decode_attn_workspace_size(params, 0) <= 8 << 20  # a split plan
    ref = pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                          window=w.window, max_seq_len=L)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = [_static(pkg, w, err) for _ in range(2)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for out in outs:
        assert torch.equal(out, ref)
    _assert_close_to_oracle(outs[1], w)


def test_static_scratch_after_a_call_that_gave_up(pkg):
    """A call whose consumers' first wait runs out (the library's
    DECODE_ATTN_TEST_STALL_TX hook makes the first stage expect more bytes
    than arrive) reports DECODE_ATTN_DEV_TIMEOUT; the next call on the
    shared array must again equal decode_attn bit for bit, with no error."""
    w = workloads.make("llama", device=DEV)
    ref = pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                          max_seq_len=w.max_seq_len())
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    os.environ["DECODE_ATTN_TEST_STALL_TX"] = "64"
    try:
        _static(pkg, w, err)
        torch.cuda.synchronize()
    finally:
        del os.environ["DECODE_ATTN_TEST_STALL_TX"]
    assert int(err.item()) & pkg.DEV_TIMEOUT
    err.zero_()
    out = _static(pkg, w, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, ref)


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
