"""Hand-derived overwrite streams on the low-bit layout of
``configs.lowbit_pair`` (packed e2m1 values and e4m3 scales whose gate/up
rows the receiver pairs in groups of 2), with the receiver bytes each must
produce, written out literally.  From the stream format (OVERWRITE records:
u32 count, u16 unit offsets, pad to 4, the new units; OVERWRITE_DENSE: the
chunk's new bytes) and the row-group layout (blog, Working with low-precision
RL: canonical row r of slot s lands on fused row (r // g) * 2g + s * g + r % g).

Receiver arena: fused gate/up e2m1 (8 rows of 2 bytes) at 0, fused scales
(8 rows of 2 bytes) at 256, the canonical e2m1 [2, 4] tensor at 512.
Chunks: 0 gate, 1 up, 2 gate_s, 3 up_s, 4 down.
"""
import numpy as np

from streamfmt import build_stream, overwrite_body

RECV_BYTES = 768


def dense_gate_stream(plan_hash):
    # gate rows 0, 1 -> fused rows 0, 1; gate rows 2, 3 -> fused rows 4, 5;
    # every byte keeps its two nibbles in place (low nibble = first element)
    body = [0x21, 0x43, 0x65, 0x87, 0xA9, 0xCB, 0xED, 0x0F]
    want = np.zeros(RECV_BYTES, dtype=np.uint8)
    want[:16] = [0x21, 0x43, 0x65, 0x87, 0, 0, 0, 0, 0xA9, 0xCB, 0xED, 0x0F, 0, 0, 0, 0]
    return build_stream(plan_hash, 0, 0, 5, [(4, 4, 0, 0, 8, 16, body)], flags=1), want


def record_stream(plan_hash):
    # up (slot 1) byte units 1 and 6: (row 0, byte 1) -> fused row 2, byte 5;
    # (row 3, byte 0) -> fused row (3 // 2) * 4 + 2 + 1 = 7, byte 14.
    # up_s (slot 1, arena byte 256) units 0 and 7: (row 0, col 0) -> fused
    # row 2 -> byte 260; (row 3, col 1) -> fused row 7 -> byte 271.
    # down (canonical, arena byte 512) units 0 and 3.
    frames = [(3, 4, 0, 1, 8, 4, overwrite_body([1, 6], [0x5A, 0xC3], 1)),
              (3, 8, 0, 3, 8, 2, overwrite_body([0, 7], [0x11, 0x77], 1)),
              (3, 4, 0, 4, 4, 3, overwrite_body([0, 3], [0xF1, 0x2E], 1))]
    want = np.zeros(RECV_BYTES, dtype=np.uint8)
    want[5], want[14] = 0x5A, 0xC3
    want[260], want[271] = 0x11, 0x77
    want[512], want[515] = 0xF1, 0x2E
    return build_stream(plan_hash, 0, 0, 5, frames, flags=1), want
