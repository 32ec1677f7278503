"""GGUF container: the oracle's layout code pinned to hand-assembled files, the library's
reader and writer checked against both, malformed files rejected, and (on a GPU) weights
read from a synthetic GGUF file multiplied by syn_mul_mat against the oracle."""
import os
import struct

import numpy as np
import pytest

from conftest import ROOT
from oracle import gguf_layout as G

GOLDEN = os.path.join(ROOT, "tests", "golden", "gguf_tiny.txt")


def golden_files():
    files, cur = {}, None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            cur = line[1:-1]
            files[cur] = b""
            continue
        files[cur] += bytes.fromhex(line.replace(" ", ""))
    return files


# the content of the two golden files, as the oracle and the writer take it
A_KV = [(b"general.architecture", G.STRING, b"llama")]
A_TENSORS = [(b"w", 0, [2], struct.pack("<2f", 1.0, 2.0))]
Q8_BLOCK = bytes([0x00, 0x3C]) + bytes(range(32))
B_KV = [(b"general.alignment", G.UINT32, 64), (b"t.arr", G.ARRAY, (G.INT32, [-1, 2, 300]))]
B_TENSORS = [(b"a", 8, [32, 1], Q8_BLOCK), (b"b", 0, [1], struct.pack("<f", -0.5))]


@pytest.fixture(scope="module")
def syn():
    import torch  # noqa: F401  (loads the CUDA runtime libsyn links against)
    from gguf_block_quantized_gb300 import build
    build.build()
    from gguf_block_quantized_gb300 import syn as s
    return s


def write(tmp_path, name, data):
    p = tmp_path / name
    p.write_bytes(data)
    return str(p)


# ---------------------------------------------------------------------------------------
# the oracle against the hand-assembled bytes
# ---------------------------------------------------------------------------------------

def test_golden_sizes_are_the_hand_computed_ones():
    f = golden_files()
    assert len(f["file_a"]) == 136 and len(f["file_b"]) == 260


def test_oracle_serializes_the_golden_files():
    f = golden_files()
    assert G.serialize(A_KV, A_TENSORS) == f["file_a"]
    assert G.serialize(B_KV, B_TENSORS, alignment=64) == f["file_b"]


def test_oracle_parses_the_golden_files():
    f = golden_files()
    a = G.parse(f["file_a"])
    assert a["version"] == 3 and a["alignment"] == 32 and a["data_start"] == 128
    assert a["kv"] == A_KV
    assert a["tensors"] == [{"name": b"w", "ne": [2], "type": 0, "offset": 0}]
    assert G.tensor_bytes(f["file_a"], a, b"w") == struct.pack("<2f", 1.0, 2.0)
    b = G.parse(f["file_b"])
    assert b["alignment"] == 64 and b["data_start"] == 192
    assert b["kv"][1] == (b"t.arr", G.ARRAY, (G.INT32, [-1, 2, 300]))
    assert [t["offset"] for t in b["tensors"]] == [0, 64]
    assert G.tensor_bytes(f["file_b"], b, b"a") == Q8_BLOCK


def test_oracle_q8_0_block_from_the_file_dequantizes_to_its_codes():
    """The Q8_0 block of file_b (d = 1.0, q = 0..31) read back through the oracle's
    dequantizer gives w = d*q = 0..31, the format table's formula."""
    import oracle
    f = golden_files()
    blk = np.frombuffer(G.tensor_bytes(f["file_b"], G.parse(f["file_b"]), b"a"), np.uint8)
    np.testing.assert_array_equal(oracle.dequantize(oracle.Q8_0, blk.reshape(1, 34), 32)[0], np.arange(32.0))


def test_oracle_rejects_bad_alignment_and_magic():
    f = golden_files()
    bad = bytearray(f["file_b"])
    bad[53:57] = struct.pack("<I", 12)  # general.alignment = 12, not a multiple of 8
    with pytest.raises(ValueError):
        G.parse(bytes(bad))
    with pytest.raises(ValueError):
        G.parse(b"GGUG" + f["file_a"][4:])


# ---------------------------------------------------------------------------------------
# the library's reader and writer
# ---------------------------------------------------------------------------------------

def test_reader_on_golden_file_a(syn, tmp_path):
    with syn.GGUFReader(write(tmp_path, "a.gguf", golden_files()["file_a"])) as r:
        assert (r.version, r.n_kv, r.n_tensors, r.alignment, r.data_start) == (3, 1, 1, 32, 128)
        assert r.get_string("general.architecture") == b"llama"
        assert r.kv_info(0) == ("general.architecture", syn.GGUF_STRING, 0, 0)
        t = r.tensor(0)
        assert (t["name"], t["ggml_type"], t["ne"], t["offset"], t["nbytes"]) == ("w", syn.GGML_F32, [2], 0, 8)
        assert t["data"].tobytes() == struct.pack("<2f", 1.0, 2.0)
        assert r.find("w") == 0 and r.find("x") == -1
        with pytest.raises(syn.SynError) as e:
            r.matrix("w")  # F32 is not a mul_mat weight format
        assert e.value.status == syn.ERR_TYPE
        with pytest.raises(syn.SynError) as e:
            r.get_int("general.architecture")
        assert e.value.status == syn.ERR_TYPE
        with pytest.raises(syn.SynError) as e:
            r.get_int("missing.key")
        assert e.value.status == syn.ERR_NOTFOUND


def test_reader_on_golden_file_b(syn, tmp_path):
    with syn.GGUFReader(write(tmp_path, "b.gguf", golden_files()["file_b"])) as r:
        assert (r.n_kv, r.n_tensors, r.alignment, r.data_start) == (2, 2, 64, 192)
        assert r.get_int("general.alignment") == 64
        et, n, p = r.get_array("t.arr")
        assert (et, n) == (syn.GGUF_INT32, 3)
        assert np.frombuffer(__import__("ctypes").string_at(p, 12), "<i4").tolist() == [-1, 2, 300]
        assert r.kv_info(1) == ("t.arr", syn.GGUF_ARRAY, syn.GGUF_INT32, 3)
        a, b = r.tensor(0), r.tensor(1)
        assert (a["ne"], a["offset"], a["nbytes"], b["offset"], b["nbytes"]) == ([32, 1], 0, 34, 64, 4)
        assert a["data"].tobytes() == Q8_BLOCK and b["data"].tobytes() == struct.pack("<f", -0.5)
        assert r.matrix("a")[:3] == (syn.Q8_0, 1, 32)
        # mapped tensor data sit at data_start + offset of the file, aligned to 64
        assert (a["data"].ctypes.data % 64, b["data"].ctypes.data % 64) == (0, 0)


def test_writer_reproduces_the_golden_files(syn, tmp_path):
    f = golden_files()
    pa = str(tmp_path / "wa.gguf")
    w = syn.GGUFWriter(pa)
    w.kv_string("general.architecture", b"llama")
    w.add_tensor("w", syn.GGML_F32, [2], np.array([1.0, 2.0], np.float32))
    w.finish()
    assert open(pa, "rb").read() == f["file_a"]
    pb = str(tmp_path / "wb.gguf")
    w = syn.GGUFWriter(pb, alignment=64)  # writes general.alignment first
    w.kv_array("t.arr", syn.GGUF_INT32, np.array([-1, 2, 300], np.int32))
    w.add_tensor("a", syn.GGML_Q8_0, [32, 1], np.frombuffer(Q8_BLOCK, np.uint8))
    w.add_tensor("b", syn.GGML_F32, [1], np.array([-0.5], np.float32))
    w.finish()
    assert open(pb, "rb").read() == f["file_b"]


def random_content(rng):
    """Random metadata of every value type and tensors of every sizable element type."""
    import oracle
    kv = [(b"general.alignment", G.UINT32, 64)]
    ints = [(G.UINT8, 0, 255), (G.INT8, -128, 127), (G.UINT16, 0, 65535), (G.INT16, -32768, 32767),
            (G.UINT32, 0, 2**32 - 1), (G.INT32, -2**31, 2**31 - 1), (G.UINT64, 0, 2**63 - 1),
            (G.INT64, -2**63, 2**63 - 1)]
    for k, (t, lo, hi) in enumerate(ints):
        kv.append((f"i.{k}".encode(), t, int(rng.integers(lo, hi, endpoint=True))))
    kv.append((b"b.true", G.BOOL, True))
    kv.append((b"f.32", G.FLOAT32, float(np.float32(rng.standard_normal()))))
    kv.append((b"f.64", G.FLOAT64, float(rng.standard_normal())))
    kv.append((b"s.empty", G.STRING, b""))
    kv.append((b"s.utf8", G.STRING, "préfill ✓".encode()))
    kv.append((b"arr.u8", G.ARRAY, (G.UINT8, [int(v) for v in rng.integers(0, 256, 7)])))
    kv.append((b"arr.f32", G.ARRAY, (G.FLOAT32, [float(np.float32(v)) for v in rng.standard_normal(5)])))
    kv.append((b"arr.str", G.ARRAY, (G.STRING, [b"<s>", b"", b"token"])))
    kv.append((b"arr.empty", G.ARRAY, (G.INT64, [])))
    tensors = []
    for name, code, n_in, n_out in [("blk.0.ffn_up.weight", 12, 512, 3), ("blk.0.ffn_down.weight", 14, 256, 5),
                                    ("blk.0.attn_q.weight", 8, 96, 4), ("blk.0.attn_k.weight", 2, 64, 2),
                                    ("blk.0.attn_v.weight", 6, 160, 3), ("output.weight", 1, 24, 2)]:
        t = {12: oracle.Q4_K, 14: oracle.Q6_K, 8: oracle.Q8_0, 2: oracle.Q4_0, 6: oracle.Q5_0, 1: oracle.F16}[code]
        q = oracle.quantize(t, rng.standard_normal((n_out, n_in)).astype(np.float32))
        tensors.append((name.encode(), code, [n_in, n_out], q.tobytes()))
    tensors.append((b"output_norm.weight", 0, [48], rng.standard_normal(48).astype("<f4").tobytes()))
    tensors.append((b"rope.bf16", 30, [3, 2, 2], rng.integers(0, 65536, 12).astype("<u2").tobytes()))
    return kv, tensors


def write_with_library(syn, path, kv, tensors, alignment):
    w = syn.GGUFWriter(path, alignment=alignment)
    for key, t, v in kv:
        k = key.decode()
        if key == b"general.alignment":
            continue
        if t == G.STRING:
            w.kv_string(k, v)
        elif t in (G.FLOAT32, G.FLOAT64):
            w.kv_float(k, t, v)
        elif t == G.ARRAY:
            et, items = v
            if et == G.STRING:
                w.kv_string_array(k, items)
            else:
                dt = {G.UINT8: "<u1", G.FLOAT32: "<f4", G.INT64: "<i8"}[et]
                w.kv_array(k, et, np.array(items, dt))
        else:
            w.kv_int(k, t, v)
    for name, code, ne, blob in tensors:
        w.add_tensor(name.decode(), code, ne, np.frombuffer(blob, np.uint8))
    w.finish()


def test_writer_and_reader_agree_with_the_oracle_on_random_content(syn, tmp_path):
    rng = np.random.default_rng(20261202)
    kv, tensors = random_content(rng)
    path = str(tmp_path / "r.gguf")
    write_with_library(syn, path, kv, tensors, 64)
    data = open(path, "rb").read()
    assert data == G.serialize(kv, tensors, alignment=64)
    p = G.parse(data)
    with syn.GGUFReader(path) as r:
        assert (r.n_kv, r.n_tensors, r.alignment, r.data_start) == (len(kv), len(tensors), 64, p["data_start"])
        for i, (key, t, v) in enumerate(kv):
            k = key.decode()
            info = r.kv_info(i)
            assert info[:2] == (k, t)
            if t == G.STRING:
                assert r.get_string(k) == v
            elif t in (G.FLOAT32, G.FLOAT64):
                assert r.get_float(k) == v
            elif t == G.ARRAY:
                et, items = v
                assert info[2:] == (et, len(items))
                if et == G.STRING:
                    assert [r.get_array_string(k, j) for j in range(len(items))] == items
                    with pytest.raises(syn.SynError):
                        r.get_array_string(k, len(items))
                elif items:
                    _, n, ptr = r.get_array(k)
                    dt = {G.UINT8: "<u1", G.FLOAT32: "<f4", G.INT64: "<i8"}[et]
                    raw = __import__("ctypes").string_at(ptr, n * np.dtype(dt).itemsize)
                    assert np.frombuffer(raw, dt).tolist() == items
            else:
                assert r.get_int(k) == v
        for i, (name, code, ne, blob) in enumerate(tensors):
            t = r.tensor(i)
            assert (t["name"], t["ggml_type"], t["ne"]) == (name.decode(), code, ne)
            assert t["offset"] == p["tensors"][i]["offset"] and t["offset"] % 64 == 0
            assert t["data"].tobytes() == blob == G.tensor_bytes(data, p, name)
            if code in (1, 2, 6, 8, 12, 14):
                typ, n_out, n_in, _, nb = r.matrix(name.decode())
                assert (n_in, n_out, nb) == (ne[0], int(np.prod(ne[1:])), len(blob))
                assert nb == n_out * syn.row_bytes(typ, n_in)


def test_reader_rejects_every_truncation(syn, tmp_path):
    f = golden_files()["file_b"]
    for n in range(0, len(f)):
        st = __import__("ctypes").c_int(0)
        h = syn.syn_gguf_open(write(tmp_path, "t.gguf", f[:n]).encode(), __import__("ctypes").byref(st))
        assert not h and st.value == syn.ERR_FORMAT, n


def patched(data, at, raw):
    b = bytearray(data)
    b[at:at + len(raw)] = raw
    return bytes(b)


@pytest.mark.parametrize("what", ["magic", "version1", "version4", "alignment12", "alignment0", "alignment_u64",
                                  "misaligned_offset", "offset_past_end", "n_dims0", "n_dims5", "ne0",
                                  "ragged_row", "value_type99", "array_of_arrays", "kv_count", "dup_key",
                                  "dup_tensor", "huge_string"])
def test_reader_rejects_malformed_files(syn, tmp_path, what):
    import ctypes
    f = golden_files()["file_b"]
    bad = {
        "magic": patched(f, 0, b"GGUG"),
        "version1": patched(f, 4, struct.pack("<I", 1)),
        "version4": patched(f, 4, struct.pack("<I", 4)),
        "alignment12": patched(f, 53, struct.pack("<I", 12)),
        "alignment0": patched(f, 53, struct.pack("<I", 0)),
        "alignment_u64": G.serialize([(b"general.alignment", G.UINT64, 64)], []),
        "misaligned_offset": patched(f, 164, struct.pack("<Q", 40)),
        "offset_past_end": patched(f, 164, struct.pack("<Q", 128)),
        "n_dims0": patched(f, 107, struct.pack("<I", 0)),
        "n_dims5": patched(f, 107, struct.pack("<I", 5)),
        "ne0": patched(f, 111, struct.pack("<Q", 0)),
        "ragged_row": patched(f, 111, struct.pack("<Q", 33)),
        "value_type99": patched(f, 70, struct.pack("<I", 99)),
        "array_of_arrays": patched(f, 74, struct.pack("<I", G.ARRAY)),
        "kv_count": patched(f, 16, struct.pack("<Q", 3)),
        "dup_key": G.serialize([(b"k", G.UINT8, 1), (b"k", G.UINT8, 2)], []),
        "dup_tensor": G.serialize([], [(b"t", 0, [1], b"\0" * 4), (b"t", 0, [1], b"\0" * 4)]),
        "huge_string": patched(f, 24, struct.pack("<Q", 2**63)),
    }[what]
    st = ctypes.c_int(0)
    assert not syn.syn_gguf_open(write(tmp_path, "bad.gguf", bad).encode(), ctypes.byref(st))
    assert st.value == syn.ERR_FORMAT


def test_reader_keeps_tensors_of_unsized_types(syn, tmp_path):
    """A tensor of an element type the reader cannot size (Q5_K, code 13) is listed with
    nbytes -1 and no data; mul_mat and upload refuse it."""
    data = G.serialize([], [(b"q5k", 13, [256, 2], b"\0" * 352), (b"f", 0, [1], b"\0" * 4)])
    with syn.GGUFReader(write(tmp_path, "u.gguf", data)) as r:
        t = r.tensor(0)
        assert (t["ggml_type"], t["nbytes"], t["data"]) == (13, -1, None)
        assert r.tensor(1)["nbytes"] == 4
        with pytest.raises(syn.SynError) as e:
            r.matrix("q5k")
        assert e.value.status == syn.ERR_TYPE
        assert syn.syn_gguf_upload(r.h, 0, 1 << 20, 1 << 20, None) == syn.ERR_TYPE


def test_open_errors(syn, tmp_path):
    import ctypes
    st = ctypes.c_int(0)
    assert not syn.syn_gguf_open(str(tmp_path / "missing.gguf").encode(), ctypes.byref(st))
    assert st.value == syn.ERR_IO
    assert not syn.syn_gguf_open(None, ctypes.byref(st)) and st.value == syn.ERR_NULL
    assert not syn.syn_gguf_open(write(tmp_path, "short.gguf", b"GGUF\3\0\0\0").encode(), ctypes.byref(st))
    assert st.value == syn.ERR_FORMAT
    assert syn.syn_gguf_n_tensors(None) == -1 and syn.syn_gguf_alignment(None) == -1
    syn.syn_gguf_close(None)


def test_upload_argument_checks_need_no_gpu(syn, tmp_path):
    with syn.GGUFReader(write(tmp_path, "b.gguf", golden_files()["file_b"])) as r:
        assert syn.syn_gguf_upload(r.h, 0, None, 64, None) == syn.ERR_NULL
        assert syn.syn_gguf_upload(r.h, 7, 1 << 20, 64, None) == syn.ERR_NOTFOUND
        assert syn.syn_gguf_upload(r.h, 0, 1 << 20, 33, None) == syn.ERR_SHAPE  # 34 bytes needed


def test_writer_errors(syn, tmp_path):
    p = str(tmp_path / "w.gguf")
    assert not syn.syn_gguf_writer_begin(p.encode(), 12)
    assert not syn.syn_gguf_writer_begin(p.encode(), 0)
    w = syn.GGUFWriter(p)
    with pytest.raises(syn.SynError):
        w.kv_int("general.alignment", syn.GGUF_UINT32, 64)  # only through the constructor
    w.kv_int("k", syn.GGUF_UINT8, 1)
    with pytest.raises(syn.SynError):
        w.kv_int("k", syn.GGUF_UINT8, 2)  # repeated key
    with pytest.raises(syn.SynError):
        w.kv_int("f", syn.GGUF_FLOAT32, 1)  # a float through the integer call
    with pytest.raises(syn.SynError):
        w.kv_float("g", syn.GGUF_INT32, 1.0)
    with pytest.raises(syn.SynError):
        w.add_tensor("t", syn.GGML_Q8_0, [33, 1], np.zeros(34, np.uint8))  # ragged row
    with pytest.raises(syn.SynError):
        w.add_tensor("t", syn.GGML_Q8_0, [32, 1], np.zeros(33, np.uint8))  # wrong byte count
    with pytest.raises(syn.SynError):
        w.add_tensor("t", 13, [256, 1], np.zeros(176, np.uint8))  # a type the reader cannot size
    w.add_tensor("t", syn.GGML_Q8_0, [32, 1], np.zeros(34, np.uint8))
    with pytest.raises(syn.SynError):
        w.add_tensor("t", syn.GGML_Q8_0, [32, 1], np.zeros(34, np.uint8))  # repeated name
    w.abort()
    assert not os.path.exists(p)
    w = syn.GGUFWriter(str(tmp_path / "no_such_dir" / "x.gguf"))
    with pytest.raises(syn.SynError) as e:
        w.finish()
    assert e.value.status == syn.ERR_IO


def test_empty_file_round_trip(syn, tmp_path):
    p = str(tmp_path / "e.gguf")
    syn.GGUFWriter(p).finish()
    data = open(p, "rb").read()
    assert data == G.serialize([], []) and len(data) == 32  # header + padding to 32
    with syn.GGUFReader(p) as r:
        assert (r.n_kv, r.n_tensors, r.data_start) == (0, 0, 32)


# ---------------------------------------------------------------------------------------
# mul_mat on weights read from a GGUF file
# ---------------------------------------------------------------------------------------

@pytest.mark.gpu
@pytest.mark.parametrize("n_tok", [1, 5, 160])
def test_mul_mat_on_weights_from_a_gguf_file(syn, tmp_path, n_tok):
    """Every weight tensor of a synthetic GGUF file (ggml names and ne = [n_in, n_out]),
    taken through syn_gguf_matrix + syn_gguf_upload into syn_mul_mat, against the oracle's
    product of the same bytes (tolerance of the oracle parity tests)."""
    import torch
    import oracle
    rng = np.random.default_rng(7 + n_tok)
    kv, _ = random_content(rng)
    shapes = [("blk.0.ffn_up.weight", G.GGML_CODE["Q4_K"], oracle.Q4_K, 1024, 136),
              ("blk.0.ffn_down.weight", G.GGML_CODE["Q6_K"], oracle.Q6_K, 512, 200),
              ("blk.0.attn_q.weight", G.GGML_CODE["Q8_0"], oracle.Q8_0, 384, 130),
              ("blk.0.attn_k.weight", G.GGML_CODE["Q4_0"], oracle.Q4_0, 320, 70),
              ("blk.0.attn_v.weight", G.GGML_CODE["Q5_0"], oracle.Q5_0, 288, 66),
              ("output.weight", G.GGML_CODE["F16"], oracle.F16, 256, 129)]
    tensors, qs = [], {}
    for name, code, t, n_in, n_out in shapes:
        q = oracle.quantize(t, rng.standard_normal((n_out, n_in)).astype(np.float32))
        qs[name] = q
        tensors.append((name.encode(), code, [n_in, n_out], q.tobytes()))
    path = str(tmp_path / "m.gguf")
    write_with_library(syn, path, kv[1:9], tensors, 32)
    with syn.GGUFReader(path) as r:
        for name, code, t, n_in, n_out in shapes:
            typ, m_out, m_in, _, nb = r.matrix(name)
            assert (typ, m_out, m_in, nb) == (t, n_out, n_in, qs[name].nbytes)
            W = r.upload(name)
            X = rng.standard_normal((n_tok, n_in)).astype(np.float32)
            Y = syn.mul_mat(typ, W, n_out, n_in, torch.from_numpy(X).cuda()).cpu().numpy().astype(np.float64)
            torch.cuda.synchronize()
            assert np.array_equal(W.cpu().numpy(), qs[name].reshape(-1))
            ref = oracle.mul_mat(t, qs[name], n_out, n_in, X)
            deq = oracle.dequantize(t, qs[name], n_in).astype(np.float64)
            bound = 1e-4 * np.linalg.norm(deq, axis=1)[None, :] * np.linalg.norm(X.astype(np.float64), axis=1)[:, None]
            assert np.all(np.abs(Y - ref) <= bound), name


def test_reader_survives_fuzzed_files(syn, tmp_path):
    """Random corruptions of valid files (byte flips, overwritten length and count fields,
    truncations, appended garbage): the reader returns either a handle or SYN_ERR_FORMAT,
    never reads outside the mapping (a crash would end the test process), and every tensor of
    a file it accepts lies inside the file."""
    import ctypes
    rng = np.random.default_rng(4242)
    kv, tensors = random_content(rng)
    base = G.serialize(kv, tensors, alignment=64)
    golden = golden_files()
    seeds = [base, golden["file_a"], golden["file_b"]]
    path = str(tmp_path / "fuzz.gguf")
    opened = 0
    for it in range(1500):
        data = bytearray(seeds[it % len(seeds)])
        kind = it % 5
        if kind == 0:  # flip a few random bytes
            for _ in range(int(rng.integers(1, 8))):
                data[int(rng.integers(0, len(data)))] ^= int(rng.integers(1, 256))
        elif kind == 1:  # overwrite a u64 at a random 8-aligned header/metadata position
            at = int(rng.integers(0, min(len(data) - 8, 512)))
            vals = [0, 1, 2**31, 2**32, 2**40, 2**63, 2**64 - 1]
            data[at:at + 8] = struct.pack("<Q", vals[int(rng.integers(0, len(vals)))])
        elif kind == 2:  # truncate
            del data[int(rng.integers(0, len(data))):]
        elif kind == 3:  # append garbage
            data += bytes(rng.integers(0, 256, int(rng.integers(1, 200))).astype(np.uint8))
        else:  # overwrite a u32 (types, dimension counts, alignment)
            at = int(rng.integers(0, min(len(data) - 4, 512)))
            vals = [0, 1, 4, 5, 9, 13, 99, 2**31]
            data[at:at + 4] = struct.pack("<I", vals[int(rng.integers(0, len(vals)))])
        with open(path, "wb") as f:
            f.write(bytes(data))
        st = ctypes.c_int(0)
        h = syn.syn_gguf_open(path.encode(), ctypes.byref(st))
        if not h:
            assert st.value == syn.ERR_FORMAT, (it, st.value)
            continue
        opened += 1
        try:
            n = syn.syn_gguf_n_tensors(h)
            ds = syn.syn_gguf_data_start(h)
            for i in range(n):
                nb, off = ctypes.c_int64(), ctypes.c_uint64()
                assert syn.syn_gguf_tensor_info(h, i, None, None, None, None, ctypes.byref(off), None,
                                                ctypes.byref(nb)) == syn.OK
                if nb.value >= 0:
                    assert ds + off.value + nb.value <= len(data)
            for i in range(syn.syn_gguf_n_kv(h)):
                assert syn.syn_gguf_kv_info(h, i, None, None, None, None) == syn.OK
        finally:
            syn.syn_gguf_close(h)
    assert opened > 0
