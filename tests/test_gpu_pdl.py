"""Dependent launches change when a kernel starts, never what it computes: a layer
step run with MOE_PDL=0 (plain stream order, in a child process) writes the same
output bits as with dependent launches (this process)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from conftest import ROOT

pytestmark = pytest.mark.gpu

STEP = r'''
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
from combine_dp_gather_gb300 import moe_dp as md, synth

spec = synth.LayerSpec("pdl", [24, 0, 70, 5, 130], synth.PAD_MAX, H=512, E=16, k=4, I=256,
                       dtype="bf16", w_std=0.05, zipf_s=1.1)
x = synth.hidden_states(spec, "cuda")
lg = synth.router_logits(spec, "cuda")
wgu, wd = synth.expert_weights(spec, device="cuda")
_, rows = md.moe_dp_layout(spec.counts, spec.mode)
layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu, w_down=wd,
                    max_rows=rows, mode=spec.mode, fp8={fp8})
out = [torch.empty(c, spec.H, device="cuda", dtype=torch.bfloat16) for c in spec.counts]
layer.forward(x, lg, out, counts=spec.counts)
torch.cuda.synchronize()
assert int(layer.status.item()) == 0
bits = torch.cat([t.view(torch.int16) for t in out]).cpu().numpy()
np.save({path!r}, bits)
'''


@pytest.mark.parametrize("fp8", [False, True])
def test_same_bits_without_dependent_launches(tmp_path, fp8):
    from combine_dp_gather_gb300 import build, moe_dp
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    moe_dp.lib()
    here, child = str(tmp_path / "on.npy"), str(tmp_path / "off.npy")
    exec(STEP.format(root=ROOT, path=here, fp8=fp8), {})
    env = dict(os.environ, MOE_PDL="0")
    r = subprocess.run([sys.executable, "-c", STEP.format(root=ROOT, path=child, fp8=fp8)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert np.array_equal(np.load(here), np.load(child))
