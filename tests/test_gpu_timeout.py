"""A bounded wait that runs out, reported as JFA_ERR_TIMEOUT.

Every wait between the roles of a kernel (TMA producer, MMA issuer, math
warps) is bounded; when one runs out the CTA raises its abort flag and the
device error word, the other roles leave, the copies and products already
issued are drained (those waits keep the full limit), tensor memory is
freed and the kernel returns.  This test builds a copy of the library whose
role waits give up after one cycle (so nearly every wait that is not
satisfied at once runs out), runs a small self-attention forward and
backward on it in a fresh process, and expects JFA_ERR_TIMEOUT from
jfa_sync_and_check.  The same process then runs the normal library, whose
results must still match the fp64 oracle: the context stays usable.
Nothing here faults or traps the GPU; the failure is a status word.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import ctypes, json, sys
sys.path.insert(0, sys.argv[1])
import torch
import jagged_flash_attention_gb300 as jfa
from jagged_flash_attention_gb300 import build
from tests.gpu_common import compare, inputs, run_gpu, run_oracle

short = ctypes.CDLL(build.variant_path("shortwait"))
P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
short.jfa_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P]
short.jfa_bwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, P, P, P]
short.jfa_sync_and_check.argtypes = [P]
short.jfa_last_error.restype = ctypes.c_char_p
x = inputs("tiny_self")
dev = torch.device("cuda")
q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
off = torch.from_numpy(x["offsets"]).to(dev)
T, H, D = q.shape
B, ml, sc = x["B"], x["max_len"], x["scale"]
out = torch.zeros_like(q)
lse = torch.zeros(H, T, device=dev)
dq, dk, dv = (torch.zeros_like(q) for _ in range(3))
s = torch.cuda.current_stream().cuda_stream
st_f = short.jfa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), off.data_ptr(), B, H, D, ml, 0, 0,
                     sc, out.data_ptr(), lse.data_ptr(), s)
st_b = short.jfa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), off.data_ptr(), B, H, D, ml, 0, 0,
                     sc, out.data_ptr(), lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                     dk.data_ptr(), dv.data_ptr(), s)
st_sync = short.jfa_sync_and_check(s)
msg = short.jfa_last_error().decode()
# the normal library on the same device and process
rep = compare(run_gpu(x), run_oracle(x))
print(json.dumps({"launch": [st_f, st_b], "sync": st_sync, "msg": msg, "normal": rep}))
"""


def test_role_wait_timeout_is_reported_and_context_survives():
    from jagged_flash_attention_gb300 import build
    build.build(variant="shortwait", defines=("JFA_ROLE_WAIT_LIMIT_CYCLES=1",))
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["launch"] == [0, 0]  # launches succeed; the device reports the timeout
    assert res["sync"] == 4, res  # JFA_ERR_TIMEOUT
    assert "bounded wait" in res["msg"]
    assert res["normal"]["out"] < 1e-2
