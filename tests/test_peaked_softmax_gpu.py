"""Peaked softmax on valid inputs: logits whose row maximum runs from 8 to
about 50, so that one or a few keys carry almost all the weight.

The tensor-core kernels round P to f16 for the PV product.  With one dominant
key the output is that key's V row; it stays exact only if the row sum is
taken over the same rounded values as the product (the weights are then
rounded P over its own sum, a convex combination).  These cases sweep the
maximum logit with a ramp over the keys (k_j scaled from 0.2 to 1, so the
running maximum grows along the sequence and forces repeated rescales), for
every head dimension, causal and bidirectional, with and without the
Gemma-style cap of 50, and hold the kernels to the f16 tolerance."""
import math

import numpy as np
import pytest
import torch

import attention_split_kv_gb300 as attn
import oracle
import seeded_inputs as si
from parity_util import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

TARGETS = [8, 16, 24, 32, 40, 50]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.build()
    attn.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield
    assert attn.attn_device_status() == attn.ATTN_OK


def peaked_prefill_case(D, causal, softcap, target, seed):
    """S=300 queries over themselves, 2 query heads on 1 kv head; k_j scaled by a
    ramp 0.2 -> 1 and the scale set so that the largest logit of the case is
    about `target` (before the cap)."""
    S = 300
    pc = si.make_prefill_case(S, 2, 1, D, seed=seed, causal=causal, softcap=softcap)
    ramp = torch.linspace(0.2, 1.0, S)[:, None, None]
    pc.k = (pc.k.float() * ramp).to(torch.float16)
    raw = torch.einsum("ihd,jd->hij", pc.q.float(), pc.k[:, 0].float())
    pc.scale = float(target / raw.abs().max())
    return pc


@pytest.mark.parametrize("target", TARGETS)
@pytest.mark.parametrize("softcap", [0.0, 50.0], ids=["nocap", "cap50"])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "bidir"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_prefill_peaked(D, causal, softcap, target):
    pc = peaked_prefill_case(D, causal, softcap, target, seed=D + target + (1 if causal else 0))
    ref, ref_lse = oracle.prefill(pc)
    g = pc.to("cuda")
    lse = torch.empty((pc.seq_len, pc.n_heads), dtype=torch.float32, device="cuda")
    out = attn.prefill(g, lse_out=lse)
    torch.cuda.synchronize()
    what = "peaked prefill D=%d causal=%s cap=%g max logit %d" % (D, causal, softcap, target)
    assert_close(out.float().cpu().numpy().reshape(ref.shape), ref, what=what)
    assert_lse_close(lse.cpu().numpy().reshape(-1), ref_lse, what=what)


def peaked_decode_case(D, softcap, target, seed, page_size=0):
    """Paged or contiguous decode (f16 cache: the tensor-core kernel for D 64/128)
    whose keys carry the same 0.2 -> 1 ramp and whose largest logit is about
    `target` (before the cap)."""
    lens = [700, 37, 1200]
    c = si.make_decode_case(3, 8, 2, D, lens, seed=seed, softcap=softcap)
    ramp = torch.linspace(0.2, 1.0, c.cap)[None, :, None, None]
    c.k = (c.k.float() * ramp).to(torch.float16)
    raw = torch.einsum("bhd,btgd->bhgt", c.q.float(), c.k.float())
    c.scale = float(target / raw.abs().max())
    if page_size:
        c = si.paged_from_contiguous(c, page_size, seed=seed + 1)
    return c


@pytest.mark.parametrize("target", TARGETS)
@pytest.mark.parametrize("softcap", [0.0, 50.0], ids=["nocap", "cap50"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_decode_peaked(D, softcap, target):
    c = peaked_decode_case(D, softcap, target, seed=3 * D + target, page_size=16 if D == 64 else 0)
    ref, ref_lse = oracle.decode(c)
    g = c.to("cuda")
    lse = torch.empty((c.batch, c.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode(g, lse_out=lse, split_keys=128)
    torch.cuda.synchronize()
    what = "peaked decode D=%d cap=%g max logit %d" % (D, softcap, target)
    assert_close(out.float().cpu().numpy().reshape(ref.shape), ref, what=what)
    assert_lse_close(lse.cpu().numpy().reshape(-1), ref_lse, what=what)
