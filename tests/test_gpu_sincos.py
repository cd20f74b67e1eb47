"""The forward's cos / sin table routine (rot_sincos: Cody-Waite reduction by 2 pi, then the
hardware approximations) against CUDA's sincosf on the same float angles."""
import ctypes
import math
import os
import shutil
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_rotation_sincos_against_sincosf(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = str(tmp_path / "sincos_check.so")
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler",
                           "-fPIC", os.path.join(HERE, "gpu_kernels", "sincos_check.cu"), "-o", so])
    lib = ctypes.CDLL(so)
    g = torch.Generator().manual_seed(0)
    special = [0.0, math.pi, -math.pi, math.pi / 2, 2 * math.pi, 1e3 * 2 * math.pi, -777.5, 2e4, -2e4]
    x = torch.cat([torch.linspace(-2e4, 2e4, 1 << 20), torch.tensor(special),
                   torch.randn(1 << 16, generator=g) * 10, torch.cumsum(torch.rand(4096, generator=g) * 0.6 - 0.3, 0)])
    x = x.float().cuda()
    out = torch.empty(x.numel() * 4, device="cuda")
    assert lib.sincos_check(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()), x.numel()) == 0
    o = out.view(-1, 4).double().cpu()
    err_s = float((o[:, 0] - o[:, 2]).abs().max())
    err_c = float((o[:, 1] - o[:, 3]).abs().max())
    assert err_s < 2e-6 and err_c < 2e-6, (err_s, err_c)
