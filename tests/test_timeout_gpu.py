"""The bounded-wait failure path, made to run without a GPU fault.

Every mbarrier wait in the kernels gives up after a limit of SM clock cycles
(about 2 s), raises its CTA's abort flag, records a timeout in the device
status word, and the CTA unwinds: copies and MMAs already issued are waited
for, tensor memory is freed, the kernel returns.  To make that path run,
this test builds a copy of the library with the limit lowered to 64 cycles
(-DNEA_WAIT_TEST=64; the product build keeps the long limit), so that the
ordinary waits for the first TMA loads run out; nothing is dropped or
corrupted on purpose.  In a child process it runs the forward, the backward,
the deterministic backward and decode through that copy and checks that each
reports NEA_ERR_TIMEOUT, then, in the same CUDA context, runs the default
library and checks its results against the fp64 oracle: the context stayed
usable.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[2])
import oracle
from causal_gqa_flashattention_gb300 import nea
from causal_gqa_flashattention_gb300.workloads import (DECODE_WORKLOADS, custom,
                                                       make_decode_inputs, make_inputs)

def rel_l2(a, ref):
    a = a.detach().float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(a - ref) / np.linalg.norm(ref))

dev = torch.device("cuda:0")
w = custom(1, 4, 2, 384, 64)
q, k, v, do = make_inputs(w, seed=11, device=dev)
o, lse = nea.attn_fwd(q, k, v, scale=w.scale)
torch.cuda.synchronize()
out = {"before": nea.check_status()}
default = nea.use_library(nea.load_library(sys.argv[1]))  # the short-wait build
nea.attn_fwd(q, k, v, scale=w.scale)
out["fwd"] = nea.check_status()
nea.attn_bwd(q, k, v, o, do, lse, scale=w.scale)
out["bwd"] = nea.check_status()
nea.attn_bwd(q, k, v, o, do, lse, scale=w.scale, deterministic=True)
out["bwd_deterministic"] = nea.check_status()
dw = DECODE_WORKLOADS["decode_gpt2s_bf16"]
dq_, kc, vc, lens = make_decode_inputs(dw, seed=0, device=dev)
nea.attn_decode(dq_, kc, vc, lens)
out["decode"] = nea.check_status()
nea.use_library(default)
o2, lse2 = nea.attn_fwd(q, k, v, scale=w.scale)
dq, dk, dv = nea.attn_bwd(q, k, v, o2, do, lse2, scale=w.scale)
torch.cuda.synchronize()
out["after"] = nea.check_status()
ro, _ = oracle.attn_fwd(q.cpu(), k.cpu(), v.cpu(), w.scale, True)
rdq, rdk, rdv = oracle.attn_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), w.scale, True)
out["o_maxabs"] = float(np.abs(o2.float().cpu().numpy() - ro).max())
out["grad_rel"] = max(rel_l2(dq, rdq), rel_l2(dk, rdk), rel_l2(dv, rdv))
print("RESULT " + json.dumps(out))
"""


def test_waits_time_out_and_unwind(cuda_device):
    from causal_gqa_flashattention_gb300 import build, nea
    build.build()
    variant = build.build_variant("waittest", ["-DNEA_WAIT_TEST=64"])
    r = subprocess.run([sys.executable, "-c", CHILD, variant, ROOT], capture_output=True,
                       text=True, timeout=600)
    lines = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")]
    assert r.returncode == 0 and lines, r.stdout[-2000:] + r.stderr[-2000:]
    out = json.loads(lines[-1][len("RESULT "):])
    assert out["before"] == nea.NEA_OK
    for what in ("fwd", "bwd", "bwd_deterministic", "decode"):
        assert out[what] == nea.NEA_ERR_TIMEOUT, (what, out)
    assert out["after"] == nea.NEA_OK
    assert out["o_maxabs"] <= 2e-2 and out["grad_rel"] <= 1e-2, out
