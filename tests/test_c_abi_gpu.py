"""The C ABI used from plain C: tests/c_abi_example.c allocates its own
device buffers with cudaMalloc, calls the fused loss (forward, backward) and
the top-K cache through include/kd.h, and writes its inputs and outputs. The
same calls through the Python binding on those inputs must give bitwise the
same results (the library is deterministic)."""

import os
import subprocess

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
T, D, V, K, CHUNK = 300, 128, 3000, 16, 64  # as in c_abi_example.c


def _load(d, name, dtype, shape):
    return np.fromfile(os.path.join(d, name), dtype=dtype).reshape(shape)


def test_c_program_matches_the_python_binding(cuda_dev, tmp_path):
    lib = os.path.join(ROOT, "top_kl_loss_tcgen05_b300", "lib")
    exe = str(tmp_path / "c_abi_example")
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), os.path.join(HERE, "c_abi_example.c"), "-o", exe,
                    "-L", lib, "-lkd", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    "-Wl,-rpath," + lib, "-Wl,-rpath," + os.path.join(CUDA, "lib64")], check=True)
    out = tmp_path / "out"
    out.mkdir()
    r = subprocess.run([exe, str(out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr

    dev = cuda_dev
    H = torch.from_numpy(_load(out, "H.bin", np.int16, (T, D))).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(_load(out, "W.bin", np.int16, (V, D))).view(torch.bfloat16).to(dev)
    ids = torch.from_numpy(_load(out, "ids.bin", np.int32, (T, K))).to(dev)
    logp = torch.from_numpy(_load(out, "logp.bin", np.float32, (T, K))).to(dev)
    x = torch.from_numpy(_load(out, "x.bin", np.float32, (T, V))).to(dev)
    scale = float(np.float32(1.0) / np.float32(T))  # the C program's 1.0f / T
    loss, lse, _ = kd.fused_kl_fwd(H, W, ids, logp, CHUNK)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, CHUNK, scale)
    tk_ids, tk_logp = kd.topk_cache(x, K)
    torch.cuda.synchronize()
    assert np.array_equal(loss.cpu().numpy().reshape(1), _load(out, "loss.bin", np.float32, (1,)))
    assert np.array_equal(lse.cpu().numpy(), _load(out, "lse.bin", np.float32, (T,)))
    assert np.array_equal(dH.cpu().numpy(), _load(out, "dH.bin", np.float32, (T, D)))
    assert np.array_equal(dW.cpu().numpy(), _load(out, "dW.bin", np.float32, (V, D)))
    assert np.array_equal(tk_ids.cpu().numpy(), _load(out, "tk_ids.bin", np.int32, (T, K)))
    assert np.array_equal(tk_logp.cpu().numpy(), _load(out, "tk_logp.bin", np.float32, (T, K)))
    assert float(loss) > 0
