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


# ---- the native reader (nt_file_*), host-only --------------------------------

def _written(tmp_path, name="tiny_q4_k_m"):
    from block_quantized_gemv_nt_gb300 import modelfile
    spec = synth.model_spec(name)
    hm = synth.make_host_model(spec, with_kv=False)
    path = tmp_path / "m.ntq"
    modelfile.write_model(str(path), spec, hm)
    return spec, hm, path


def _split(data: bytes):
    """(header dict, data section) of a file's bytes."""
    import json
    import struct
    hlen = struct.unpack("<Q", data[8:16])[0]
    data0 = (16 + hlen + 4095) // 4096 * 4096
    return json.loads(data[16:16 + hlen]), data[data0:]


def _join(header, body: bytes, version=1, raw=None) -> bytes:
    """A file with header `header` (or the literal text `raw`) in front of data section `body`."""
    import json
    import struct
    h = raw if raw is not None else json.dumps(header).encode()
    pre = b"NTQF" + struct.pack("<IQ", version, len(h)) + h
    return pre + bytes((-len(pre)) % 4096) + body


@pytest.mark.parametrize("name", ["tiny_q4_k_m", "tiny_f16"])
def test_native_reader_matches_writer(tmp_path, name):
    """nt_file_open reads back what the writer laid out: the descriptor (the
    runtime fields zero), the header text, and every entry's offset, size and
    bytes in the mapping."""
    import ctypes
    from block_quantized_gemv_nt_gb300 import engine, modelfile, nt
    spec, hm, path = _written(tmp_path, name)
    f = nt.nt_file_open(str(path))
    try:
        d, want = nt.nt_file_desc(f), engine.model_desc(spec)
        for fld, _ in nt.nt_model_desc._fields_:
            if fld in ("kv_cap", "stream_slots"):
                assert getattr(d, fld) == 0
            else:
                assert getattr(d, fld) == getattr(want, fld), fld
        data = path.read_bytes()
        header, _ = _split(data)
        assert nt.nt_file_header(f) == data[16:16 + len(nt.nt_file_header(f))].decode()
        data0 = (16 + len(nt.nt_file_header(f)) + 4095) // 4096 * 4096
        for ename, (rel, n) in header["entries"].items():
            addr, off, nbytes = nt.nt_file_entry(f, ename)
            assert (off, nbytes) == (data0 + rel, n), ename
            assert ctypes.string_at(addr, n) == data[off:off + n], ename
        addr, off, n = nt.nt_file_entry(f, "blob.1")
        wq = np.ascontiguousarray(hm.layers[1]["wq"])
        assert ctypes.string_at(addr, wq.nbytes) == wq.tobytes()
        with pytest.raises(nt.NtError):
            nt.nt_file_entry(f, "blob.999")
    finally:
        nt.nt_file_close(f)
    mf = modelfile.ModelFile(str(path))   # the Python views agree with the native offsets
    assert np.array_equal(mf.layers[1]["wq"], hm.layers[1]["wq"])
    mf.close()


def test_native_reader_json(tmp_path):
    """The header's JSON reader takes what RFC 8259 allows (escapes, a
    surrogate pair, nested values, literals, exponents) and refuses what it
    does not, each with a reason on the calling thread."""
    from block_quantized_gemv_nt_gb300 import nt
    _, _, path = _written(tmp_path)
    header, body = _split(path.read_bytes())
    ok = dict(header)
    ok["note"] = ["café \U0001F600 \"q\" \\ /\t", {"a": [True, False, None, -0.5e-3, 12, []]}, {}]
    p = tmp_path / "ok.ntq"
    p.write_bytes(_join(ok, body))
    f = nt.nt_file_open(str(p))
    import json
    assert json.loads(nt.nt_file_header(f))["note"] == ok["note"]
    nt.nt_file_close(f)
    text = path.read_bytes()[16:16 + len(json.dumps(header).encode())]
    bad = {
        "trailing comma": text[:-1] + b",}",
        "unterminated string": b'{"spec": "abc',
        "lone low surrogate": text[:-1] + b', "x": "\\udc00"}',
        "bare control char": text[:-1] + b', "x": "a\x01b"}',
        "leading zero": text[:-1] + b', "x": 012}',
        "not an object": b"[1, 2]",
        "nested too deep": text[:-1] + b', "x": ' + b"[" * 100 + b"]" * 100 + b"}",
        "trailing garbage": text + b" x",
    }
    for why, raw in bad.items():
        p = tmp_path / "bad.ntq"
        p.write_bytes(_join(None, body, raw=raw))
        with pytest.raises(nt.NtError) as ei:
            nt.nt_file_open(str(p))
        assert ei.value.status == nt.NT_ERR_INVALID_ARG, why
        assert str(p) in str(ei.value), why
        assert ("not a JSON object" if why == "not an object" else "not valid JSON") in str(ei.value), why


def test_native_reader_refusals(tmp_path):
    """Each check of nt_file_open refuses a file that breaks it, before any
    entry is handed out: version, blob layout, entry alignment, a missing or
    wrongly sized entry, a duplicate, an entry past the end, a format id."""
    import copy
    from block_quantized_gemv_nt_gb300 import nt
    _, _, path = _written(tmp_path)
    header, body = _split(path.read_bytes())

    def edited(fn):
        h = copy.deepcopy(header)
        fn(h)
        return _join(h, body)

    cases = {
        "version": _join(header, body, version=2),
        "blob layout": edited(lambda h: h["blob_offsets"].__setitem__(1, h["blob_offsets"][1] + 256)),
        "blob bytes": edited(lambda h: h.__setitem__("blob_bytes", h["blob_bytes"] + 256)),
        "misaligned": edited(lambda h: h["entries"]["out"].__setitem__(0, h["entries"]["out"][0] + 16)),
        "missing": edited(lambda h: h["entries"].pop("ffn_norm.1")),
        "norm size": edited(lambda h: h["entries"]["attn_norm.0"].__setitem__(1, 4)),
        "embd size": edited(lambda h: h["entries"]["embd"].__setitem__(1, h["entries"]["embd"][1] - 1)),
        "short blob": edited(lambda h: h["entries"]["blob.0"].__setitem__(1, h["blob_bytes"] - 1)),
        "past the end": edited(lambda h: h["entries"]["out"].__setitem__(0, len(body))),
        "negative": edited(lambda h: h["entries"]["out"].__setitem__(0, -4096)),
        "format id": edited(lambda h: h["spec"]["fmt"].__setitem__("wq", 7)),
        "ragged": edited(lambda h: h["spec"].__setitem__("d_model", h["spec"]["d_model"] + 32)),
        "gqa": edited(lambda h: h["spec"].__setitem__("n_kvh", h["spec"]["n_qh"] + 1)),
        "no eps": edited(lambda h: h["spec"].pop("eps")),
        "float dim": edited(lambda h: h["spec"].__setitem__("n_layers", 2.0)),
    }
    raw_dup = _join(header, body).replace(b'"entries": {', b'"entries": {"out": [0, 4], ', 1)
    import struct
    hl = struct.unpack("<Q", raw_dup[8:16])[0] + len(b'"out": [0, 4], ')
    cases["duplicate"] = _join(None, body, raw=raw_dup[16:16 + hl])
    for why, data in cases.items():
        p = tmp_path / "bad.ntq"
        p.write_bytes(data)
        with pytest.raises(nt.NtError) as ei:
            nt.nt_file_open(str(p))
        assert ei.value.status == nt.NT_ERR_INVALID_ARG, why
    p = tmp_path / "good.ntq"
    p.write_bytes(_join(header, body))
    nt.nt_file_close(nt.nt_file_open(str(p)))   # the unedited header still opens
    with pytest.raises(nt.NtError):
        nt.nt_file_open(str(tmp_path / "absent.ntq"))
    with pytest.raises(nt.NtError):
        nt.nt_file_open(str(tmp_path))          # a directory
    assert nt.lib().nt_file_close(None) == nt.NT_ERR_INVALID_ARG


def test_native_reader_survives_mutated_headers(tmp_path):
    """The reader meets untrusted bytes: 1500 seeded mutations of a valid
    header (bytes overwritten, inserted, deleted; digits changed; the header
    length field off by one or by a page) each either open — and then every
    entry lies inside the file, 4096-aligned — or are refused with a reason;
    none crashes the process.  The data section stays in place."""
    import os
    import struct
    from block_quantized_gemv_nt_gb300 import nt
    _, _, path = _written(tmp_path, "tiny_q4_0")
    data = path.read_bytes()
    size = len(data)
    hlen = struct.unpack("<Q", data[8:16])[0]
    data0 = (16 + hlen + 4095) // 4096 * 4096
    head = bytes(data[16:16 + hlen])
    rng = np.random.default_rng(20240611)
    alphabet = b'{}[]":,.-+eE0123456789 \\untrfalsx'
    opened = refused = 0
    fd = os.open(str(path), os.O_RDWR)
    try:
        for _ in range(1500):
            h = bytearray(head)
            for _ in range(int(rng.integers(1, 4))):
                i = int(rng.integers(0, len(h)))
                op = int(rng.integers(0, 4))
                c = alphabet[int(rng.integers(0, len(alphabet)))]
                if op == 0:
                    h[i] = c
                elif op == 1:
                    h.insert(i, c)
                elif op == 2 and len(h) > 1:
                    del h[i]
                elif chr(h[i]).isdigit():
                    h[i] = ord("0") + int(rng.integers(0, 10))
            n = max(0, len(h) + int(rng.choice([0, 0, 0, -1, 1, 4096])))
            pre = b"NTQF" + struct.pack("<IQ", 1, n) + bytes(h)
            if len(pre) > data0:
                continue
            os.pwrite(fd, pre + bytes(data0 - len(pre)), 0)
            try:
                f = nt.nt_file_open(str(path))
            except nt.NtError as e:
                assert e.status == nt.NT_ERR_INVALID_ARG and str(path) in str(e)
                refused += 1
                continue
            for name in ("embd", "out", "out_norm", "blob.0", "attn_norm.2", "ffn_norm.2"):
                _, off, nbytes = nt.nt_file_entry(f, name)
                assert off % 4096 == 0 and off + nbytes <= size
            nt.nt_file_close(f)
            opened += 1
    finally:
        os.close(fd)
    print(f"mutated headers: {opened} opened, {refused} refused")
    assert opened > 0 and refused > 0


def test_refuse_in_place_hook_arguments():
    """The rung-order test hook takes 0 or 1 only (host-side state, no GPU)."""
    from block_quantized_gemv_nt_gb300 import nt
    assert nt.lib().nt_debug_file_refuse_in_place(2) == nt.NT_ERR_INVALID_ARG
    assert nt.lib().nt_debug_file_refuse_in_place(-1) == nt.NT_ERR_INVALID_ARG
    nt.nt_debug_file_refuse_in_place(True)
    nt.nt_debug_file_refuse_in_place(False)
