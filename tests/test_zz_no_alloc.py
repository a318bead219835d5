"""attn_decode_noalloc: decode for callers that cannot allocate device memory
(an engine plugin with no allocator, a decode loop that must never call
cudaMalloc).  It takes its scratch from a fixed device array inside the
library, so its results must equal those of attn_decode given a caller
workspace.  This file is collected last (its name sorts after every other test
file), so a run that stops at the first failure has run everything else first;
it needs no state from earlier tests and also passes alone in a fresh process:
python -m pytest tests/test_zz_no_alloc.py -m gpu"""
import numpy as np
import pytest
import torch

import attention_split_kv_gb300 as attn
import seeded_inputs as si
from parity_util import assert_close

pytestmark = pytest.mark.gpu


def _noalloc(g, out, lse, split_keys=0):
    attn.attn_decode_noalloc(g.q, g.k, g.v, g.kv_len, g.page_table, g.page_size, g.max_pages, g.n_pages,
                             g.cap, g.k_scales, g.v_scales, attn.ATTN_KV_INT8 if g.int8 else attn.ATTN_KV_F16,
                             g.batch, g.n_heads, g.n_kv_heads, g.head_dim, g.window, g.softcap, g.scale,
                             split_keys, out, lse)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    attn.build()
    attn.load()
    cases = [si.make_decode_case(4, 8, 2, 128, (1, 900), seed=301, page_size=16),
             si.make_decode_case(3, 16, 4, 64, [700, 5, 1500], seed=302, int8=True, window=600)]
    for case in cases:
        g = case.to("cuda")
        ref_lse = torch.empty((g.batch, g.n_heads), dtype=torch.float32, device="cuda")
        ref = attn.decode(g, lse_out=ref_lse)
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        _noalloc(g, out, lse)
        torch.cuda.synchronize()
        assert_close(out.float().cpu().numpy(), ref.double().cpu().numpy(), int8=g.int8, what="noalloc")
        assert np.allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=2e-3, rtol=0, equal_nan=False)
    assert attn.attn_device_status() == attn.ATTN_OK


def test_noalloc_smaller_call_after_a_larger_one():
    # every call shares the one scratch array, which keeps the previous call's
    # contents: a smaller call (same head_dim and layout) after a larger one must
    # still read only what it wrote itself
    attn.load()
    big = si.make_decode_case(8, 32, 8, 128, (2000, 4900), seed=311, page_size=16).to("cuda")
    small = si.make_decode_case(2, 8, 2, 128, [300, 1200], seed=312, page_size=16).to("cuda")
    out_big = torch.empty((big.batch, big.n_heads, big.head_dim), dtype=torch.float16, device="cuda")
    _noalloc(big, out_big, None)
    ref_lse = torch.empty((small.batch, small.n_heads), dtype=torch.float32, device="cuda")
    ref = attn.decode(small, lse_out=ref_lse)
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    _noalloc(small, out, lse)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(lse, ref_lse)
    assert attn.attn_device_status() == attn.ATTN_OK


def test_noalloc_rejects_sizes_above_its_fixed_scratch():
    attn.load()
    B, Hq, Hkv, D, max_kv = 4096, 64, 8, 256, 32768
    assert attn.attn_decode_workspace_size(B, Hq, Hkv, D, max_kv) > (16 << 20)
    q = torch.empty((1,), dtype=torch.float16, device="cuda")
    with pytest.raises(attn.AttnError) as ei:
        attn.attn_decode_noalloc(q, q, q, q, None, 0, 0, 0, max_kv, None, None, attn.ATTN_KV_F16, B, Hq, Hkv, D,
                                 0, 0.0, 0.125, 0, q, None)
    assert ei.value.status == attn.ATTN_EUNSUPPORTED
    assert "16777216" in str(ei.value)
