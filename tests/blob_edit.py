"""Byte-level edits of NWC blobs for robustness tests (no decoding arithmetic here).

Layout facts used: header fields n_blocks at byte 24 and data offset at byte 48 and total size
at byte 56 (u64), the u32 block table at byte 80 in 16-byte units from the data section, and a
block region that starts with 32 u8 lane word counts followed by the code words and a zero pad
to 16 bytes.
"""
import numpy as np


def region_bounds(blob, i):
    a = np.frombuffer(bytes(blob), np.uint8)
    nb = int(a[24:32].view(np.uint64)[0])
    off_data = int(a[48:56].view(np.uint64)[0])
    tab = a[80:80 + 4 * (nb + 1)].view(np.uint32)
    return off_data + 16 * int(tab[i]), off_data + 16 * int(tab[i + 1])


def replace_code_streams(blob, i, lane_words, word=0xFFFFFFFF):
    """The blob with block i's code streams replaced: lane l gets lane_words[l] copies of `word`
    (each count at most 26, so host validation still accepts the region); the block's raw
    section and escape list are kept, and the block table and total size follow the new size."""
    assert len(lane_words) == 32 and all(0 <= w <= 26 for w in lane_words)
    a = bytearray(blob)
    start, end = region_bounds(blob, i)
    old_codes = 4 * sum(a[start:start + 32])
    tail = bytes(a[start + ((32 + old_codes + 15) // 16) * 16:end])  # raw section + escape list
    codes = np.full(sum(lane_words), word, np.uint32).astype("<u4").tobytes()
    head = bytes(lane_words) + codes
    head += b"\0" * (-len(head) % 16)
    region = head + tail
    delta = len(region) - (end - start)
    assert delta % 16 == 0
    out = bytearray(a[:start]) + region + bytearray(a[end:])
    nb = int(np.frombuffer(bytes(out[24:32]), np.uint64)[0])
    tab = np.frombuffer(bytes(out[80:80 + 4 * (nb + 1)]), np.uint32).copy()
    tab[i + 1:] += delta // 16
    out[80:80 + 4 * (nb + 1)] = tab.astype("<u4").tobytes()
    total = int(np.frombuffer(bytes(out[56:64]), np.uint64)[0]) + delta
    out[56:64] = np.array([total], "<u8").tobytes()
    return bytes(out)
