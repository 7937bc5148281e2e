"""Patch files (host only): round trip, the kilobyte-scale size of a
100-entry patch, and rejection of corrupted files."""
import pytest

from bit_weight_gemv_sign_b300 import patchfile, synth


def test_round_trip_of_the_27b_patch(tmp_path):
    entries = synth.patch_entries_27b(100, 0)
    path = tmp_path / "bankai.patch"
    n = patchfile.save(str(path), entries)
    assert n == 8 + 4 + 7 * 100 == 712      # about a kilobyte, like the pages' patches
    assert patchfile.load(str(path)) == [tuple(e) for e in entries]


def test_empty_patch():
    assert patchfile.decode(patchfile.encode([])) == []


@pytest.mark.parametrize("mutate", ["magic", "short", "long", "count"])
def test_corrupted_files_are_rejected(mutate):
    data = bytearray(patchfile.encode([(1, 2, 3), (63, 6, 17407)]))
    if mutate == "magic":
        data[0] ^= 0xFF
    elif mutate == "short":
        data = data[:-1]
    elif mutate == "long":
        data += b"\x00"
    else:
        data[8] += 1
    with pytest.raises(patchfile.PatchFileError):
        patchfile.decode(bytes(data))


def test_out_of_range_entries_are_rejected():
    with pytest.raises(patchfile.PatchFileError):
        patchfile.encode([(70000, 0, 0)])
    with pytest.raises(patchfile.PatchFileError):
        patchfile.encode([(0, 300, 0)])
    with pytest.raises(patchfile.PatchFileError):
        patchfile.encode([(0, 0, -1)])
