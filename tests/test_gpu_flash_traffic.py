"""Regression check of the flash-attention kernel's DRAM traffic (GPU, opt-in).

The prefill attention kernel dispatches its CTAs in L2-sized bands of (sequence, kv group)
pairs so that the CTAs resident together share K/V tiles through L2; that order is how the
hardware dispatches a 1-D grid, observed rather than guaranteed.  If it ever changes, K and V
are re-read from DRAM and the kernel's DRAM reads grow above the bytes it must read once: the
rotated queries, keys and values.  This test measures one launch's dram__bytes_read.sum with
ncu (one metric, one pass, clocks left alone) on B=4 x T=8192 and checks it stays within 5 %
of those bytes.  It runs only with GQA_NCU_CHECK=1 (it profiles a child process) and needs
ncu on PATH.
"""
import csv
import io
import os
import shutil
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from transformer_gqa_attention_gb300 import _build, abi
from transformer_gqa_attention_gb300 import inputs as gin
_build.build()
B, T = 4, 8192
inp = gin.make_custom(seed=2, B=B, T=T)
ctx = abi.attn_create(*[t.cuda() for t in (inp.wq, inp.wk, inp.wv, inp.wo)])
x, R = inp.x.cuda(), inp.R.cuda()
ck = torch.zeros(B, T, 8, 128, dtype=torch.bfloat16, device="cuda"); cv = torch.zeros_like(ck)
d = torch.empty(B, T, 4096, dtype=torch.float32, device="cuda")
flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
for _ in range(2):
    flush.zero_()
    abi.attn_prefill(ctx, x, B, T, R, True, ck, cv, T, 0, d)
abi.attn_sync_status(ctx)
abi.attn_destroy(ctx)
"""


@pytest.mark.skipif(os.environ.get("GQA_NCU_CHECK") != "1" or shutil.which("ncu") is None,
                    reason="opt-in ncu check (GQA_NCU_CHECK=1, ncu on PATH)")
def test_flash_reads_each_q_k_v_byte_once():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cmd = [sys.executable, "-c", CHILD, ROOT]
    subprocess.run(cmd, check=True, timeout=600)  # the same command exits 0 without ncu first
    out = subprocess.run(["ncu", "--metrics", "dram__bytes_read.sum", "--clock-control", "none",
                          "-k", "regex:flash_prefill", "-s", "1", "-c", "1", "--csv", *cmd],
                         check=True, timeout=600, capture_output=True, text=True).stdout
    rows = [r for r in csv.reader(io.StringIO(out[out.index('"ID"'):])) if len(r) > 5]
    hdr = rows[0]
    vals = [r for r in rows[1:] if r[hdr.index("Metric Name")] == "dram__bytes_read.sum"]
    assert len(vals) == 1
    unit = vals[0][hdr.index("Metric Unit")]
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}[unit]
    read = float(vals[0][hdr.index("Metric Value")].replace(",", "")) * scale
    unique = 4 * 8192 * (4096 + 1024 + 1024) * 2  # Q_r, K_r, V (bf16), each once
    assert abs(read / unique - 1) < 0.05, f"flash DRAM reads {read / 1e6:.1f} MB vs {unique / 1e6:.1f} MB unique"
