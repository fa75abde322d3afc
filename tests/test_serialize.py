"""State files (host side): round trip for every moment mode, the pages' flags (both
moments compressed / a quantized v follows), and rejection of damaged or mismatched files."""
import io
import os

import pytest
import torch


@pytest.fixture(scope="module")
def psa():
    import __graft_entry__
    __graft_entry__.build()
    import precision_state_adam_gb300 as psa
    return psa


def _random_state(mode, sizes, seed=0):
    g = torch.Generator().manual_seed(seed)
    nb = lambda n: (n + 2047) // 2048
    if mode == "fp32":
        return ([torch.randn(n, generator=g) for n in sizes], [torch.rand(n, generator=g) for n in sizes])
    if mode == "bf16m":
        return ([torch.randn(n, generator=g).bfloat16() for n in sizes],
                [torch.rand(n, generator=g).bfloat16() for n in sizes])
    if mode == "q8":
        return ([torch.randint(-127, 128, (n,), generator=g, dtype=torch.int8) for n in sizes],
                [torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8) for n in sizes],
                [torch.rand(nb(n), generator=g) for n in sizes], [torch.rand(nb(n), generator=g) for n in sizes])
    return ([torch.randn(n, generator=g) for n in sizes],
            [torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8) for n in sizes],
            [torch.rand(nb(n), generator=g) for n in sizes])


@pytest.mark.parametrize("mode", ["fp32", "bf16m", "q8", "q8v"])
def test_round_trip_is_bit_exact(psa, mode, tmp_path):
    sizes = [1, 2047, 2049, 5000, 0]
    st = _random_state(mode, sizes)
    path = os.path.join(tmp_path, "state.bin")
    psa.save_state(path, mode, st, step=17, hparams={"lr": 1e-3}, q8={"percentile": 99.9})
    mode2, st2, step, header = psa.load_state(path)
    assert mode2 == mode and step == 17 and header["hparams"]["lr"] == 1e-3
    assert header["compress_both_moments"] == (mode == "q8")
    assert header["has_v_quantized"] == (mode in ("q8", "q8v"))
    for a_part, b_part in zip(st, st2):
        for a, b in zip(a_part, b_part):
            assert a.dtype == b.dtype and a.shape == b.shape
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b)


def test_damaged_and_mismatched_files_are_rejected(psa):
    st = _random_state("q8", [3000])
    buf = io.BytesIO()
    psa.save_state(buf, "q8", st, step=2)
    data = bytearray(buf.getvalue())
    flipped = bytearray(data)
    flipped[len(flipped) // 2] ^= 0x40
    with pytest.raises(psa.StateFormatError, match="checksum"):
        psa.load_state(io.BytesIO(bytes(flipped)))
    with pytest.raises(psa.StateFormatError, match="not a psadam"):
        psa.load_state(io.BytesIO(b"XXXXXXXX" + bytes(data[8:])))
    with pytest.raises(ValueError):
        psa.save_state(io.BytesIO(), "q8", st[:3], step=1)  # a part is missing
    with pytest.raises(ValueError):
        bad = (st[0], st[1], st[2], [torch.zeros(5)])  # wrong scale count
        psa.save_state(io.BytesIO(), "q8", bad, step=1)


@pytest.mark.parametrize("mode", ["q8", "q8v"])
def test_round_trip_other_block_size(psa, mode):
    sizes = [1, 300, 1000]
    bs = 256
    g = torch.Generator().manual_seed(5)
    nb = lambda n: (n + bs - 1) // bs
    if mode == "q8":
        st = ([torch.randint(-127, 128, (n,), generator=g, dtype=torch.int8) for n in sizes],
              [torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8) for n in sizes],
              [torch.rand(nb(n), generator=g) for n in sizes], [torch.rand(nb(n), generator=g) for n in sizes])
    else:
        st = ([torch.randn(n, generator=g) for n in sizes],
              [torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8) for n in sizes],
              [torch.rand(nb(n), generator=g) for n in sizes])
    buf = io.BytesIO()
    psa.save_state(buf, mode, st, step=3, block_size=bs)
    buf.seek(0)
    mode2, st2, step, header = psa.load_state(buf)
    assert header["block_size"] == bs and mode2 == mode and step == 3
    for a_part, b_part in zip(st, st2):
        for a, b in zip(a_part, b_part):
            assert torch.equal(a, b)
    with pytest.raises(ValueError):  # scales sized for the default block
        psa.save_state(io.BytesIO(), mode, st, step=3)


def _forge(header_bytes: bytes, body: bytes = b"") -> io.BytesIO:
    import struct
    import zlib
    blob = b"PSADAMST" + struct.pack("<II", 1, len(header_bytes)) + header_bytes + body
    return io.BytesIO(blob + struct.pack("<I", zlib.crc32(blob) & 0xFFFFFFFF))


def test_malformed_headers_are_format_errors(psa):
    # files whose checksum is right but whose header is not a valid state header
    import json
    good = {"mode": "fp32", "step": 1, "block_size": 2048, "compress_both_moments": False,
            "has_v_quantized": False, "hparams": {}, "q8": {}, "numel": [2],
            "arrays": [["0.m", "f32", 2], ["0.v", "f32", 2]]}
    body = bytes(16)
    mode, st, step, _ = psa.load_state(_forge(json.dumps(good).encode(), body))
    assert mode == "fp32" and step == 1 and st[0][0].numel() == 2
    cases = [
        b"not json",
        b"[1, 2, 3]",                                         # not an object
        json.dumps({k: v for k, v in good.items() if k != "numel"}).encode(),
        json.dumps({**good, "numel": [-4]}).encode(),
        json.dumps({**good, "numel": "2"}).encode(),
        json.dumps({**good, "arrays": [["0.m", "f32", 2]]}).encode(),        # one array short
        json.dumps({**good, "arrays": [["0.m", "f32", 2], ["0.v", "f32"]]}).encode(),
        json.dumps({**good, "mode": "q4"}).encode(),
        json.dumps({**good, "block_size": 0}).encode(),
        json.dumps({**good, "has_v_quantized": True}).encode(),
        json.dumps({**good, "step": "x"}).encode(),
    ]
    for hb in cases:
        with pytest.raises(psa.StateFormatError):
            psa.load_state(_forge(hb, body))
    with pytest.raises(psa.StateFormatError, match="truncated"):
        psa.load_state(_forge(json.dumps(good).encode(), body[:12]))
    with pytest.raises(psa.StateFormatError, match="trailing"):
        psa.load_state(_forge(json.dumps(good).encode(), body + b"\0"))
