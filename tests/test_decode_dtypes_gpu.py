"""GPU parity of the decode query and output element types (attn_decode_ex,
attn_decode_tiered): f32 queries on the tensor-core kernel (two f16 terms into
one accumulator) and on the CUDA-core kernel (read as f32, or 16-bit fixed
point for int8 caches), f32 outputs, and the bit-identities that tie them to
the f16 path."""
import numpy as np
import pytest
import torch

import attention_split_kv_gb300 as attn
import oracle
import seeded_inputs as si
from parity_util import assert_close, assert_lse_close, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.build()
    attn.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield
    assert attn.attn_device_status() == attn.ATTN_OK


def _run(case, out_f32, split_keys=64, tiered=False):
    g = case.to("cuda")
    lse = torch.empty((case.batch, case.n_heads), dtype=torch.float32, device="cuda")
    fn = attn.decode_tiered if tiered else attn.decode
    out = fn(g, lse_out=lse, split_keys=split_keys, out_f32=out_f32)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu().numpy()


CASES = {
    # name: (D, int8, page_size, ring) -- which split kernel and layout
    "tc_d128": (128, False, 0, 0),
    "tc_d64_paged": (64, False, 16, 0),
    "tc_d128_ring": (128, False, 0, 64),
    "cc_d256": (256, False, 0, 0),
    "cc_int8_paged": (128, True, 16, 0),
    "cc_int8_contig": (128, True, 0, 0),
    "cc_paged2": (128, False, 2, 0),
}


def _case(name, q_f32):
    D, int8, P, ring = CASES[name]
    c = si.make_decode_case(3, 8, 2, D, [5, 300, 1000], seed=D + P + ring, int8=int8, page_size=P,
                            window=700, q_f32=q_f32)
    return si.ring_from_contiguous(c, ring) if ring else c


@pytest.mark.parametrize("out_f32", [False, True], ids=["out16", "out32"])
@pytest.mark.parametrize("name", list(CASES))
def test_f32_queries_match_oracle(name, out_f32):
    c = _case(name, q_f32=True)
    assert c.q.dtype == torch.float32
    ref, ref_lse = oracle.decode(c)
    out, lse = _run(c, out_f32)
    assert out.dtype == (torch.float32 if out_f32 else torch.float16)
    assert_close(out.float().numpy().reshape(ref.shape), ref, int8=c.int8, what=name)
    assert_lse_close(lse.reshape(-1), ref_lse, what=name)


@pytest.mark.parametrize("name", list(CASES))
def test_f16_valued_f32_queries_and_f32_out_are_the_f16_path(name):
    # q in f32 holding f16 values is the same query (the tensor-core kernel's lo
    # term is zero); f32 out holds the values the f16 path rounds
    c16 = _case(name, q_f32=False)
    c32 = si.DecodeCase(**{**c16.__dict__, "q": c16.q.float()})
    a, la = _run(c16, out_f32=False)
    b, lb = _run(c32, out_f32=True)
    assert torch.equal(b.half(), a)
    assert np.array_equal(la, lb)


@pytest.mark.parametrize("name", ["tc_d128", "tc_d64_paged"])
def test_f32_queries_keep_their_precision(name):
    # against the fp64 oracle on the f32 queries, the two-term product beats
    # the same queries rounded to f16 (both with f32 out)
    c = _case(name, q_f32=True)
    ref, _ = oracle.decode(c)
    exact, _ = _run(c, out_f32=True)
    rounded, _ = _run(si.DecodeCase(**{**c.__dict__, "q": c.q.half()}), out_f32=True)
    e_exact = errors(exact.numpy().reshape(ref.shape), ref)[1]
    e_round = errors(rounded.numpy().reshape(ref.shape), ref)[1]
    assert e_exact < 0.75 * e_round, (e_exact, e_round)


@pytest.mark.parametrize("out_f32", [False, True], ids=["out16", "out32"])
def test_tiered_int8_with_f32_queries(out_f32):
    # the int8 tier of the pages takes f32 queries
    c = si.make_tiered_case(4, 8, 2, 128, [0, 300, 1000, 77], [40, 0, 200, 64], 64, seed=17, int8=True,
                            page_size=16, window=600, q_f32=True)
    ref, ref_lse = oracle.decode_tiered(c)
    out, lse = _run(c, out_f32, tiered=True)
    assert_close(out.float().numpy().reshape(ref.shape), ref, int8=True, what="tiered f32 q")
    assert_lse_close(lse.reshape(-1), ref_lse, what="tiered f32 q")
