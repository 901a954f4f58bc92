"""The C ABI from plain C: tests/c_client.c includes only ringattn.h and the CUDA
runtime's C header, links libringattn.so and libcudart, and runs ring_attn_fwd on
buffers it allocates itself. On the CPU the client must compile and link; on a GB300
its output must match the fp64 oracle and equal the Python binding's bit for bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from online_softmax_merge_gb300 import build as B
from online_softmax_merge_gb300.inputs import Workload, make_qkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client.c")
LAYOUTS = {"contiguous": 0, "striped": 1, "zigzag": 2}


def compile_client(out_dir: str) -> str:
    lib = B.build()
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(B.nvcc_path())))
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(out_dir, "c_client")
    libdir = os.path.dirname(lib)
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Werror", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-lringattn", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    exe = compile_client(str(tmp_path))
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_client_matches_oracle_and_binding(tmp_path):
    import online_softmax_merge_gb300 as ra
    from gpu_helpers import TOL_LSE, TOL_O
    from oracle.attention import dense_attention

    w = Workload("cclient", 2, 4 * (128 + 72), 4, 2, 128, 4, "striped", True, 900)
    exe = compile_client(str(tmp_path))
    q, k, v = make_qkv(w)
    for name, t in (("q", q), ("k", k), ("v", v)):
        t.contiguous().view(torch.int16).numpy().tofile(str(tmp_path / f"{name}.bin"))
    args = [str(tmp_path), w.batch, w.seqlen, w.heads, w.kv_heads, w.head_dim, w.P,
            int(w.causal), LAYOUTS[w.layout]]
    r = subprocess.run([exe] + [str(a) for a in args], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    o = torch.from_numpy(np.fromfile(str(tmp_path / "o.bin"), dtype=np.int16)).view(
        torch.bfloat16).reshape(q.shape)
    lse = torch.from_numpy(np.fromfile(str(tmp_path / "lse.bin"), dtype=np.float32)).reshape(
        w.batch, w.heads, w.seqlen)
    O, L = dense_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), True)
    assert np.abs(o.double().numpy() - O).max() <= TOL_O
    assert np.abs(lse.double().numpy() - L).max() <= TOL_LSE
    dev = torch.device("cuda:0")
    o2, l2 = ra.fwd(q.to(dev), k.to(dev), v.to(dev), w.P, w.layout, w.causal)
    torch.cuda.synchronize(dev)
    assert torch.equal(o, o2.cpu()) and torch.equal(lse, l2.cpu())
