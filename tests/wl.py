"""Test helpers: synth workloads -> library descriptors and device arenas."""
import numpy as np

import bit_exact_xor_gb300 as dcr


def descs_of(wl):
    out = []
    for t in wl.tensors:
        out.append(dcr.make_desc(t.name, t.elem_bits, t.rows, t.cols, t.split, wl.tp, t.shard_offset,
                                 t.recv_offset, t.q_heads, t.kv_heads, t.head_dim, t.recv_layout,
                                 t.recv_group, t.recv_slot))
    return out


def to_device(arrs):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(a)).to("cuda") for a in arrs]
