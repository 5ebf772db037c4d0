"""A C caller of libnt.so (tests/c/decode_file.c): the public C API
("Ntransformer" (en.unwiki.net), roadmap) used from a C program with no
Python in its process — a model file opened by the library's own reader,
resident layers uploaded from its mapping, the others page-locked in place
and streamed, a prompt prefilled and greedy steps decoded — against the fp64
oracle on the same weights.  The header compiles as strict C99."""
import glob
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "decode_file.c")


def _cuda_dirs():
    """(include dir, directory holding libcudart.so) of the toolkit nvcc belongs to."""
    from block_quantized_gemv_nt_gb300 import build
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(build._nvcc())))
    for d in [os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")] + glob.glob(os.path.join(cuda, "targets", "*", "lib")):
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return os.path.join(cuda, "include"), d
    pytest.skip("no libcudart.so next to nvcc")


def _compile(out_dir: str) -> str:
    from block_quantized_gemv_nt_gb300 import build, nt  # noqa: F401  (importing nt builds libnt.so when stale)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc, libdir = _cuda_dirs()
    so_dir = os.path.dirname(build.SO)
    exe = os.path.join(out_dir, "decode_file")
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           "-isystem", inc, SRC, "-o", exe, "-L", so_dir, "-lnt", "-L", libdir, "-lcudart",
           f"-Wl,-rpath,{so_dir}:{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_caller_compiles(tmp_path):
    """The C program builds against include/nt.h and links against libnt.so
    (strict C99, warnings as errors); run without arguments it prints its
    usage and exits 2 without touching a GPU."""
    exe = _compile(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 2 and "usage" in r.stderr


@pytest.mark.gpu
def test_c_caller_decodes_model_file(tmp_path):
    from gpu_util import need_gpu
    need_gpu()
    from block_quantized_gemv_nt_gb300 import modelfile
    spec = synth.model_spec("small_q4_k_m_r1")   # 4 layers, layer 0 resident, 1..3 streamed from the file
    hm = synth.make_host_model(spec, with_kv=False)
    path = str(tmp_path / "m.ntq")
    modelfile.write_model(path, spec, hm)
    exe = _compile(str(tmp_path))
    raw = synth.random_bytes(4 * 19, seed=spec.seed, stream=4242).view(np.uint32)
    prompt = (raw % spec.vocab).astype(np.int32)   # 19 tokens: a chunk of 16 and a ragged one of 3
    n_decode = 4
    out = str(tmp_path / "logits.f32")
    r = subprocess.run([exe, path, str(spec.n_resident), str(spec.kv_cap), str(n_decode), out,
                        *[str(int(t)) for t in prompt]], capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("streamed from the file") == spec.n_layers - spec.n_resident
    got = np.fromfile(out, dtype=np.float32).reshape(1 + n_decode, spec.vocab).astype(np.float64)
    shape = (spec.n_layers, spec.n_kvh, spec.kv_cap, spec.head_dim)
    om = oracle.Model(spec, hm.layers, hm.embd, hm.out, hm.out_norm, np.zeros(shape, np.float16),
                      np.zeros(shape, np.float16))
    for i, t in enumerate(prompt):
        ref = om.step(int(t), i)
    pos = len(prompt)
    for k, g in enumerate(got):
        if k > 0:   # teacher-forced on the program's own greedy tokens
            ref = om.step(int(np.argmax(got[k - 1])), pos)
            pos += 1
        assert np.max(np.abs(g - ref)) <= 2e-2 * ref.std(), k
        assert int(np.argmax(g)) == int(np.argmax(ref)), k
