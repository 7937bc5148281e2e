"""Row-patch files: a Bankai-style patch is a list of (layer, projection, row)
entries whose rows are XOR-flipped in place and removed by the same XOR (web
page "LocalLLaMA, true 1-bit LLM용 XOR patch 방식 "Bankai" 실험에 주목",
section "LocalLLaMA가 본 핵심 포인트": patches of about a kilobyte that name
which projection rows of which layer to flip).

File layout (little-endian): the 8-byte magic b"BIT1XPAT", a uint32 entry
count, then per entry a uint16 layer, a uint8 projection index and a uint32
row (7 bytes, packed).  100 entries take 712 bytes.
"""
from __future__ import annotations

import struct

MAGIC = b"BIT1XPAT"
_ENTRY = struct.Struct("<HBI")


class PatchFileError(ValueError):
    pass


def encode(entries) -> bytes:
    """Bytes of a patch file holding ``entries`` [(layer, projection, row), ...]."""
    out = bytearray(MAGIC)
    entries = list(entries)
    out += struct.pack("<I", len(entries))
    for layer, proj, row in entries:
        if not (0 <= layer < 1 << 16 and 0 <= proj < 1 << 8 and 0 <= row < 1 << 32):
            raise PatchFileError(f"entry out of range: {(layer, proj, row)}")
        out += _ENTRY.pack(layer, proj, row)
    return bytes(out)


def decode(data: bytes):
    """Entries of a patch file; raises PatchFileError on a bad magic, a bad
    count or trailing bytes."""
    if len(data) < len(MAGIC) + 4 or data[:len(MAGIC)] != MAGIC:
        raise PatchFileError("not a patch file")
    (count,) = struct.unpack_from("<I", data, len(MAGIC))
    body = data[len(MAGIC) + 4:]
    if len(body) != count * _ENTRY.size:
        raise PatchFileError(f"expected {count} entries ({count * _ENTRY.size} bytes), got {len(body)} bytes")
    return [_ENTRY.unpack_from(body, i * _ENTRY.size) for i in range(count)]


def save(path: str, entries) -> int:
    data = encode(entries)
    with open(path, "wb") as f:
        f.write(data)
    return len(data)


def load(path: str):
    with open(path, "rb") as f:
        return decode(f.read())
