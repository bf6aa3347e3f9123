"""GGUF interop (host, no GPU): the product's writer checked by an
independent test-side parser, round trips of q4_K / q6_K / F32 tensors
through write and read, and malformed files refused without crashing."""
import struct

import numpy as np
import pytest

from q4_q8_int8_gb300 import synthetic


def _mmq():
    import q4_q8_int8_gb300 as mmq
    from q4_q8_int8_gb300 import build
    build.build()
    mmq.load_library()
    return mmq


def _parse(path):
    """Minimal GGUF reader written from the format description (little
    endian): magic, version, counts, metadata, tensor infos, data offsets."""
    b = open(path, "rb").read()
    pos = 0

    def take(fmt):
        nonlocal pos
        v = struct.unpack_from("<" + fmt, b, pos)
        pos += struct.calcsize("<" + fmt)
        return v[0] if len(v) == 1 else v

    def string():
        nonlocal pos
        n = take("Q")
        s = b[pos:pos + n].decode()
        pos += n
        return s

    assert b[:4] == b"GGUF"
    pos = 4
    version, nt, nkv = take("I"), take("Q"), take("Q")
    meta = {}
    for _ in range(nkv):
        k, t = string(), take("I")
        assert t == 4          # the writer only emits the u32 alignment
        meta[k] = take("I")
    infos = []
    for _ in range(nt):
        name, nd = string(), take("I")
        dims = [take("Q") for _ in range(nd)]
        infos.append((name, dims, take("I"), take("Q")))
    align = meta.get("general.alignment", 32)
    data0 = (pos + align - 1) // align * align
    return version, meta, infos, data0, b


def _tensors():
    rng = np.random.default_rng(41)
    q4 = synthetic.q4K_weights(3, 512, 42)
    q6 = synthetic.q6K_weights(2, 256, 43)
    f32 = rng.standard_normal((5, 12)).astype(np.float32)
    return [("blk.0.ffn_up.weight", 12, 512, 3, q4), ("blk.0.attn_q.weight", 14, 256, 2, q6),
            ("norm.weight", 0, 12, 5, f32)]


def test_writer_bytes_by_independent_parser(tmp_path):
    mmq = _mmq()
    path = str(tmp_path / "t.gguf")
    ts = _tensors()
    mmq.gguf_write(path, ts)
    version, meta, infos, data0, b = _parse(path)
    assert version == 3 and meta == {"general.alignment": 32}
    assert [(n, d, t) for n, d, t, _ in infos] == [(t[0], [t[2], t[3]], t[1]) for t in ts]
    for (name, dims, typ, off), t in zip(infos, ts):
        assert off % 32 == 0
        raw = np.ascontiguousarray(t[4]).view(np.uint8).reshape(-1)
        assert b[data0 + off:data0 + off + raw.size] == raw.tobytes()


def test_round_trip(tmp_path):
    mmq = _mmq()
    path = str(tmp_path / "r.gguf")
    ts = _tensors()
    mmq.gguf_write(path, ts)
    got = mmq.gguf_read(path)
    assert list(got) == [t[0] for t in ts]
    for name, typ, ne0, ne1, arr in ts:
        t, dims, buf = got[name]
        assert t == typ and dims == (ne0, ne1)
        assert (buf == np.ascontiguousarray(arr).view(np.uint8).reshape(-1)).all()


def test_malformed_files_are_refused(tmp_path):
    mmq = _mmq()
    path = str(tmp_path / "m.gguf")
    mmq.gguf_write(path, _tensors())
    good = open(path, "rb").read()

    def refused(data):
        p = str(tmp_path / "bad.gguf")
        open(p, "wb").write(data)
        with pytest.raises(mmq.MMQError):
            mmq.gguf_read(p)

    _, _, infos, data0, _ = _parse(path)
    last_end = data0 + infos[-1][3] + 5 * 12 * 4            # end of the last tensor's data
    for cut in (0, 3, 4, 10, 23, 40, 60, 100, data0 + 7, last_end - 1):   # truncated anywhere
        refused(good[:cut])
    refused(b"GGUX" + good[4:])                                   # magic
    refused(good[:4] + struct.pack("<I", 9) + good[8:])           # version
    refused(good[:8] + struct.pack("<Q", 1 << 40) + good[16:])    # tensor count
    refused(good[:16] + struct.pack("<Q", 1 << 40) + good[24:])   # metadata count
    # first tensor's offset: misaligned, then past the end
    name0 = infos[0][0].encode()
    at = good.index(name0) + len(name0) + 4 + 2 * 8 + 4
    refused(good[:at] + struct.pack("<Q", 8) + good[at + 8:])
    refused(good[:at] + struct.pack("<Q", 1 << 40) + good[at + 8:])


def test_unsupported_types_are_listed_without_bytes(tmp_path):
    # a Q8_0 tensor (type 8) is listed with size 0 rather than refused
    mmq = _mmq()
    path = str(tmp_path / "u.gguf")
    mmq.gguf_write(path, _tensors()[:1])
    b = bytearray(open(path, "rb").read())
    _, _, infos, _, _ = _parse(path)
    name0 = infos[0][0].encode()
    at = bytes(b).index(name0) + len(name0) + 4 + 2 * 8
    b[at:at + 4] = struct.pack("<I", 8)
    p = str(tmp_path / "u2.gguf")
    open(p, "wb").write(bytes(b))
    got = mmq.gguf_read(p)
    t, dims, buf = got[infos[0][0]]
    assert t == 8 and buf.size == 0
