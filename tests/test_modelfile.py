"""Model files (the host-file tier): the writer's layout read back through the
mapping, byte for byte (CPU only; the GPU side is in test_stream_gpu.py)."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("name", ["tiny_q4_k_m", "tiny_f32"])
def test_roundtrip(tmp_path, name):
    from block_quantized_gemv_nt_gb300 import modelfile
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec, with_kv=False)
    path = str(tmp_path / "m.ntq")
    modelfile.write_model(path, spec, hm)
    mf = modelfile.ModelFile(path)
    assert mf.spec.n_layers == spec.n_layers and mf.spec.fmt == spec.fmt and mf.spec.kv_cap == spec.kv_cap
    assert np.array_equal(mf.embd, hm.embd) and np.array_equal(mf.out, hm.out)
    assert np.array_equal(mf.out_norm, hm.out_norm)
    for a, b in zip(mf.layers, hm.layers):
        for k in b:
            assert np.array_equal(a[k], b[k]), k
    # every entry starts on a page, and a layer's seven matrices are one range
    for name_, (off, n) in mf.entries.items():
        assert off % 4096 == 0
    off0 = mf.entries["blob.0"][0]
    assert mf.layers[0]["wq"].ctypes.data == mf._buf.ctypes.data + off0
    mf.close()


def test_rejects_other_files(tmp_path):
    from block_quantized_gemv_nt_gb300 import modelfile
    p = tmp_path / "x.bin"
    p.write_bytes(b"GGUF" + bytes(60))
    with pytest.raises(ValueError):
        modelfile.ModelFile(str(p))


def test_rejects_truncated_files(tmp_path):
    """A file cut short (past its header, inside its data) is refused before
    any entry is viewed or page-locked."""
    from block_quantized_gemv_nt_gb300 import modelfile
    spec = synth.model_spec("tiny_q8_0")
    hm = synth.make_host_model(spec, with_kv=False)
    path = tmp_path / "m.ntq"
    modelfile.write_model(str(path), spec, hm)
    data = path.read_bytes()
    for cut in (10, 40, len(data) - 4096):
        p = tmp_path / f"cut{cut}.ntq"
        p.write_bytes(data[:cut])
        with pytest.raises(ValueError):
            modelfile.ModelFile(str(p))
    modelfile.ModelFile(str(path)).close()
