"""The one-launch decode of small calls (decode_direct_kernel).

A plain decode with the automatic split plan (split_keys = 0) whose sequences
keep at most 512 keys, whose query-head group times head dim is at most 1024
and whose cache is small (at most 2^22 to 2^24 (sequence, kv head, key, dim)
elements by head dim and dtype; int8: at most 2^15 (key, dim) elements per
sequence) runs without splits and without the combine pass.  These tests compare it with the fp64 oracle over
every layout (contiguous, paged, ring), element type (f16 and int8 caches, f16
and f32 queries and outputs) and option (window, softcap), at the sizes where
the path ends, and with the split path (an explicit split_keys) on the same
inputs.  Which kernel runs is checked by the launch trace (test_trace_gpu.py);
the clamped kv_len, empty-sequence and bad-page-id cases run on both paths in
test_decode_gpu.py.
"""
import numpy as np
import pytest
import torch

import attention_split_kv_gb300 as attn
import oracle
import seeded_inputs as si
from parity_util import F16_MAX_ABS, INT8_MAX_ABS, LSE_MAX_ABS, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.build()
    attn.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield
    assert attn.attn_device_status() == attn.ATTN_OK


def _run(case, split_keys=0, max_kv=None, out_f32=False):
    g = case.to("cuda")
    lse = torch.empty((case.batch, case.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode(g, lse_out=lse, split_keys=split_keys, max_kv=max_kv, out_f32=out_f32)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check(case, what, **kw):
    ref, ref_lse = oracle.decode(case)
    got, lse = _run(case, **kw)
    assert_close(got.reshape(ref.shape), ref, int8=case.int8, what=what)
    assert_lse_close(lse.reshape(-1), ref_lse, what=what)
    return got, lse


CASES = [
    # B, Hq, Hkv, D, lens
    (1, 4, 2, 64, [128]),                  # the tiny GQA 2:1 decode
    (3, 16, 1, 64, [1, 255, 512]),         # G = 16 (G*D = 1024), a sequence at the key bound
    (2, 6, 2, 64, [250, 17]),              # G = 3
    (4, 8, 8, 128, [0, 1, 100, 256]),      # MHA, an empty and a one-key sequence
    (2, 16, 2, 128, [250, 33]),            # G = 8 (G*D = 1024)
    (2, 8, 2, 256, [120, 7]),              # D = 256, G = 4 (G*D = 1024)
    (3, 4, 4, 256, [7, 64, 128]),
]


def _layout(case, layout, seed):
    if layout == "contiguous":
        return case
    if layout.startswith("paged"):
        return si.paged_from_contiguous(case, int(layout[5:]), seed=seed)
    return si.ring_from_contiguous(case, 256)      # logical lengths up to 512 over 256 slots


@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("layout", ["contiguous", "paged1", "paged16", "ring"])
@pytest.mark.parametrize("shape", CASES, ids=lambda s: "B%d_H%d_%d_D%d" % s[:4])
def test_direct_matches_oracle(shape, layout, int8):
    if int8 and layout == "paged1":
        pytest.skip("int8 caches need pages of >= 8 tokens")
    B, Hq, Hkv, D, lens = shape
    seed = (B * 131 + Hq * 17 + D) % 997
    case = _layout(si.make_decode_case(B, Hq, Hkv, D, lens, seed=seed, int8=int8), layout, seed)
    _check(case, "direct %s %s" % (layout, shape))


@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("layout", ["contiguous", "paged16", "ring"])
def test_direct_agrees_with_the_split_path(layout, int8):
    case = _layout(si.make_decode_case(3, 8, 2, 128, [250, 64, 3], seed=5, int8=int8), layout, 5)
    a, la = _check(case, "direct " + layout)
    b, lb = _check(case, "split " + layout, split_keys=64)
    # the split path rounds p to f16 (tensor-core kernel) or q to 16-bit fixed
    # point (int8): the two agree within the parity bounds, not bit for bit
    np.testing.assert_allclose(a, b, rtol=0, atol=INT8_MAX_ABS if int8 else F16_MAX_ABS)
    np.testing.assert_allclose(la, lb, rtol=0, atol=LSE_MAX_ABS)


@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("page_size", [8, 16, 64])
def test_direct_paged_is_bit_identical_to_contiguous(page_size, int8):
    case = si.make_decode_case(3, 8, 2, 128, [5, 250, 200], seed=41, int8=int8, cap=256)
    paged = si.paged_from_contiguous(case, page_size, seed=42)
    a, la = _run(case, max_kv=256)
    b, lb = _run(paged, max_kv=256)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("window", [1, 5, 100, 512])
def test_direct_window_over_a_long_cache(window):
    # kv_len up to 1200, but a window of at most 512 keys keeps the call on the
    # direct path
    case = si.make_decode_case(3, 8, 2, 128, [50, 333, 1200], seed=51, window=window)
    _check(case, "window %d" % window)
    paged = si.make_decode_case(3, 8, 2, 64, [50, 333, 1200], seed=52, window=window, page_size=16, int8=True)
    _check(paged, "paged int8 window %d" % window)


@pytest.mark.parametrize("softcap", [1.0, 30.0])
@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
def test_direct_softcap(softcap, int8):
    case = si.make_decode_case(2, 8, 2, 128, [250, 90], seed=61, softcap=softcap, scale=0.3, int8=int8)
    _check(case, "softcap %g" % softcap)


@pytest.mark.parametrize("out_f32", [False, True], ids=["out16", "out32"])
@pytest.mark.parametrize("q_f32", [False, True], ids=["q16", "q32"])
@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
def test_direct_f32_queries_and_outputs(q_f32, out_f32, int8):
    case = si.make_decode_case(3, 8, 2, 64, [300, 1, 77], seed=71, int8=int8, q_f32=q_f32, page_size=16)
    _check(case, "q_f32=%d out_f32=%d" % (q_f32, out_f32), out_f32=out_f32)


def test_direct_peaked_logits():
    # keys ramped 0.2 -> 1 and the scale set so the largest logit is 50
    for D in (64, 128, 256):
        c = si.make_decode_case(3, 8, 2, D, [500, 37, 200], seed=D)
        ramp = torch.linspace(0.2, 1.0, c.cap)[None, :, None, None]
        c.k = (c.k.float() * ramp).to(torch.float16)
        raw = torch.einsum("bhd,btgd->bhgt", c.q.float(), c.k.float())
        c.scale = float(50.0 / raw.abs().max())
        _check(c, "peaked D=%d" % D)


def test_direct_many_sequences():
    lens = [(7 * b) % 17 for b in range(4096)]     # 0 .. 16 keys, some empty
    case = si.make_decode_case(4096, 4, 1, 64, lens, seed=4096, page_size=8)
    _check(case, "4096 sequences")


def test_direct_noalloc_equals_workspace_call():
    g = si.make_decode_case(2, 8, 2, 128, [300, 12], seed=97, page_size=16).to("cuda")
    ref_lse = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    ref = attn.decode(g, lse_out=ref_lse)
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    attn.attn_decode_noalloc(g.q, g.k, g.v, g.kv_len, g.page_table, g.page_size, g.max_pages, g.n_pages, g.cap,
                             None, None, attn.ATTN_KV_F16, 2, 8, 2, 128, 0, 0.0, g.scale, 0, out, lse)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
def test_direct_f16_valued_f32_queries_and_f32_out_are_the_f16_path(int8):
    # q in f32 holding f16 values is the same query; f32 out holds the values the
    # f16 path rounds
    c16 = si.make_decode_case(3, 8, 2, 128, [200, 1, 77], seed=73, int8=int8, page_size=16)
    c32 = si.DecodeCase(**{**c16.__dict__, "q": c16.q.float()})
    g16, g32 = c16.to("cuda"), c32.to("cuda")
    la = torch.empty((3, 8), dtype=torch.float32, device="cuda")
    lb = torch.empty((3, 8), dtype=torch.float32, device="cuda")
    a = attn.decode(g16, lse_out=la)
    b = attn.decode(g32, lse_out=lb, out_f32=True)
    torch.cuda.synchronize()
    assert b.dtype == torch.float32
    assert torch.equal(b.half(), a) and torch.equal(la, lb)
