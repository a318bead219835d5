"""ATTN_TRACE=1: every launch is described on stderr from the host (kernel,
grid, block, shared memory, split plan).  Run in a child process, since the
switch is read once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
import attention_split_kv_gb300 as attn
import seeded_inputs as si
attn.build(); attn.load()
attn.prefill(si.make_prefill_case(200, 4, 2, 64, seed=1, causal=True).to("cuda"))
attn.decode(si.make_decode_case(2, 8, 2, 128, [700, 40], seed=2, page_size=16).to("cuda"))
attn.decode(si.make_decode_case(2, 8, 2, 128, [700, 40], seed=3, int8=True).to("cuda"))
attn.decode(si.make_decode_case(1, 4, 2, 64, [128], seed=5).to("cuda"))
attn.decode(si.make_decode_case(1, 4, 2, 64, [128], seed=5).to("cuda"), split_keys=16)
attn.decode(si.make_decode_case(1, 4, 2, 64, [512], seed=6).to("cuda"))
attn.decode(si.make_decode_case(1, 4, 2, 64, [513], seed=7).to("cuda"))
attn.prefill(si.make_prefill_case(2560, 8, 4, 256, seed=4, causal=True).to("cuda"))
torch.cuda.synchronize()
assert attn.attn_device_status() == attn.ATTN_OK
"""


def _run(env_value):
    env = dict(os.environ)
    env.pop("ATTN_TRACE", None)
    if env_value is not None:
        env["ATTN_TRACE"] = env_value
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stderr.splitlines() if ln.startswith("[libattn]")]


def test_trace_describes_every_launch():
    lines = _run("1")
    text = "\n".join(lines)
    assert "prefill_tc_kernel<D=64,mode=raw,paged=0> grid=(4,2,1)" in text, text
    assert "decode_tc_kernel<D=128,NH=2,f32q=0>" in text and "layout=paged" in text, text
    assert "decode_split_kernel<D=128,int8=1,GH=4>" in text and "layout=contiguous" in text, text
    assert text.count("decode_combine_kernel<D=128,tiers=1,out=f16>") == 2, text
    assert "prefill_tc_kernel<D=256,mode=raw,paged=0> grid=(8,20,1)" in text, text
    assert "order=heads fastest, longest query tiles first" in text, text
    # small decodes: one launch, one CTA per (sequence, kv head), unless a split
    # size is given or a sequence may keep more than 512 keys (capacity 520)
    assert text.count("decode_direct_kernel<D=64,int8=0,GM=2> grid=2 block=256") == 2, text
    assert "max_keys=128" in text and "max_keys=512" in text, text
    assert text.count("decode_tc_kernel<D=64,NH=2,f32q=0>") == 2, text
    assert text.count("decode_combine_kernel<D=64,tiers=1,out=f16>") == 2, text
    assert len(lines) == 12, text


def test_trace_is_off_by_default():
    assert _run(None) == []
    assert _run("0") == []
