"""The usage file (Learn, kept between runs) and the hot-set selection, on the
host: no GPU is used.  The file layout is pinned by a file built here byte by
byte from its written description, with an independent FNV-1a."""
import os
import struct

import numpy as np
import pytest


@pytest.fixture(scope="module")
def m():
    from int4_routed_expert_sigmoid_gb300 import build
    build.build()
    import int4_routed_expert_sigmoid_gb300 as pkg
    return pkg


def fnv1a64(data: bytes) -> int:
    h = 0xCBF29CE484222325
    for b in data:
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def handmade(hits: np.ndarray, model_id: int, version: int = 1) -> bytes:
    layers, E = hits.shape
    body = b"MOEUSAGE" + struct.pack("<IIIIQ", version, layers, E, 0, model_id)
    body += b"".join(struct.pack("<Q", int(v)) for v in hits.reshape(-1))
    return body + struct.pack("<Q", fnv1a64(body))


def test_round_trip_and_byte_layout(m, tmp_path):
    rng = np.random.default_rng(0)
    hits = rng.integers(0, 2 ** 40, size=(3, 256), dtype=np.uint64)
    hits[1, 7] = 2 ** 64 - 1
    path = str(tmp_path / "layer.usage")
    m.usage_save(path, hits, model_id=0xC011B21)
    assert not os.path.exists(path + ".tmp")
    assert open(path, "rb").read() == handmade(hits, 0xC011B21)
    assert np.array_equal(m.usage_load(path, 3, 256, 0xC011B21), hits)
    # a file built by hand from the layout loads
    other = str(tmp_path / "hand.usage")
    small = np.arange(10, dtype=np.uint64).reshape(2, 5) * np.uint64(3)
    open(other, "wb").write(handmade(small, 42))
    assert np.array_equal(m.usage_load(other, 2, 5, 42), small)


def test_stale_file_is_refused(m, tmp_path):
    hits = np.ones((2, 8), np.uint64)
    path = str(tmp_path / "u")
    m.usage_save(path, hits, model_id=7)
    for layers, E, mid in ((2, 8, 8), (3, 8, 7), (2, 16, 7)):
        with pytest.raises(m.MoeError) as ei:
            m.usage_load(path, layers, E, mid)
        assert ei.value.status == m.MOE_ERR_STALE


@pytest.mark.parametrize("damage", ["flip_count", "flip_header", "truncate", "pad", "magic", "version", "missing"])
def test_damaged_file_is_refused(m, tmp_path, damage):
    hits = np.arange(32, dtype=np.uint64).reshape(4, 8)
    path = str(tmp_path / "u")
    data = bytearray(handmade(hits, 99))
    if damage == "flip_count":
        data[40] ^= 0x01
    elif damage == "flip_header":
        data[13] ^= 0x80
    elif damage == "truncate":
        data = data[:-9]
    elif damage == "pad":
        data += b"\0" * 8
    elif damage == "magic":
        data[0:8] = b"MOEUSAGX"
    elif damage == "version":
        data = bytearray(handmade(hits, 99, version=2))
    if damage != "missing":
        open(path, "wb").write(bytes(data))
    with pytest.raises(m.MoeError) as ei:
        m.usage_load(path, 4, 8, 99)
    assert ei.value.status == m.MOE_ERR_INVALID_ARG


def test_top_experts_order(m):
    rng = np.random.default_rng(3)
    for E in (1, 8, 256):
        h = rng.integers(0, 5, size=E).astype(np.uint64)   # many ties
        want = sorted(range(E), key=lambda e: (-int(h[e]), e))
        for n in {0, 1, min(8, E), E}:
            assert list(m.usage_top(h, n)) == want[:n]
    with pytest.raises(m.MoeError):
        m.usage_top(np.zeros(4, np.uint64), 5)
