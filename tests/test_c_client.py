"""The C ABI from a plain C program (tests/c_client/lazyattn_client.c): compiled
with gcc against include/lazyattn.h and liblazyattn.so, device memory from the
CUDA runtime, no Python on the path. On CPU it runs the host-only checks; on the
GPU it runs one request (ragged documents, a query segment, decode steps) whose
inputs this test writes and whose outputs it compares with the fp64 oracle.
"""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

import oracle
import workload
from tests.gpu_common import compare

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    import __graft_entry__
    __graft_entry__.build()
    from position_agnostic_kv_lazyattn_gb300 import lazyattn
    gcc = shutil.which("gcc")
    if gcc is None or not os.path.exists(os.path.join(CUDA_HOME, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA runtime headers are missing")
    libdir = os.path.dirname(lazyattn.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_client") / "lazyattn_client")
    cmd = [gcc, "-std=c99", "-O2", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA_HOME, "include"), os.path.join(ROOT, "tests", "c_client", "lazyattn_client.c"),
           "-L", libdir, "-llazyattn", "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(CUDA_HOME, "lib64"), "-o", exe]
    p = subprocess.run(cmd, capture_output=True, text=True)
    assert p.returncode == 0, p.stdout + p.stderr
    return exe


def test_c_client_host_checks(client):
    p = subprocess.run([client, "host"], capture_output=True, text=True, timeout=60)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "host checks ok" in p.stdout


def _case(dtype, hq, hkv, d, doc_lens, q_len, n_steps, seed):
    rng = np.random.default_rng(seed)

    def draw(*shape):
        x = rng.standard_normal(shape).astype(np.float32)
        return workload.round_bf16(x) if dtype == "bf16" else x

    docs = [(draw(n, hkv, d), draw(n, hkv, d)) for n in doc_lens]
    q, kq, vq = draw(q_len, hq, d), draw(q_len, hkv, d), draw(q_len, hkv, d)
    steps = [(draw(hq, d), draw(hkv, d), draw(hkv, d)) for _ in range(n_steps)]
    return docs, (q, kq, vq), steps


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,hq,hkv,d,doc_lens,q_len,n_steps",
                         [("f32", 4, 2, 64, [32, 7, 45], 16, 4),
                          ("bf16", 32, 8, 128, [40, 256, 17], 29, 5)])
def test_c_client_runs_the_path(client, tmp_path, dtype, hq, hkv, d, doc_lens, q_len, n_steps):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    theta = 1.0e4 if dtype == "f32" else 5.0e5
    docs, (q, kq, vq), steps = _case(dtype, hq, hkv, d, doc_lens, q_len, n_steps, 41)
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(src, "wb") as f:
        f.write(struct.pack("<8i", 0x4C415A59, int(dtype == "bf16"), hq, hkv, d, len(docs), q_len, n_steps))
        f.write(struct.pack("<d", theta))
        f.write(np.array(doc_lens, "<i4").tobytes())
        for k, v in docs:
            f.write(k.astype("<f4").tobytes())
            f.write(v.astype("<f4").tobytes())
        for a in (q, kq, vq):
            f.write(a.astype("<f4").tobytes())
        for st in steps:
            for a in st:
                f.write(a.astype("<f4").tobytes())
    p = subprocess.run([client, "run", str(src), str(dst)], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stdout + p.stderr
    out = np.fromfile(dst, "<f4")
    assert out.size == (q_len + n_steps) * hq * d
    pre = out[:q_len * hq * d].reshape(q_len, hq, d)
    dec = out[q_len * hq * d:].reshape(n_steps, hq, d)
    compare(pre, oracle.prefill_request(docs, q, kq, vq, theta), dtype)
    ref = oracle.decode_request(docs, kq, vq, steps, theta)
    for t in range(n_steps):
        compare(dec[t], ref[t], dtype)
