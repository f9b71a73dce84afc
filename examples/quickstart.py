"""Quickstart: encode a 1 % change of a small TP=2 model on the GPU and apply
it in place to a receiver holding the old weights, through the Python
binding over the C ABI (build first: python -c "import __graft_entry__ as g;
g.build()")."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch
import bit_exact_xor_gb300 as dcr

H, TP = 1024, 2
w_bytes = (H // TP) * H * 2                       # one bf16 shard of an [H, H] weight
arena = w_bytes + H * 2                           # + a replicated bf16 norm [H]
descs = [
    dcr.make_desc("w", 16, H, H, dcr.SPLIT_ROWS, TP, [0, 0], 0),                  # row-split shards
    dcr.make_desc("norm", 16, 1, H, dcr.REPLICATED, TP, [w_bytes, w_bytes], H * H * 2),
]
plan = dcr.Plan(descs)

g = torch.Generator(device="cuda").manual_seed(0)
old = [torch.randint(0, 256, (arena,), dtype=torch.uint8, device="cuda", generator=g) for _ in range(TP)]
new = [x.clone() for x in old]
for x in new:                                     # flip the low bit of ~1 % of the bf16 values
    v = x.view(torch.int16)
    hit = torch.rand(v.numel(), device="cuda", generator=g) < 0.01
    v[hit] = v[hit] ^ 1

# receiver: its copy of the old weights, in the checkpoint layout, at version 0
target = torch.empty(plan.info.recv_bytes, dtype=torch.uint8, device="cuda")
dcr.check(dcr.dense_refit(plan, old, target))
state = dcr.RecvState(plan, version=0)

# sender: encode version 0 -> 1
payload = torch.empty(plan.window(0).payload_bound, dtype=torch.uint8, device="cuda")
rc, size, changed = dcr.encode(plan, old, new, payload, base_version=0, target_version=1)
dcr.check(rc)

# ... payload[:size] travels to the receiver ...
rc, result = dcr.apply(plan, state, payload, size, target)
dcr.check(rc)
assert state.version == 1
assert torch.equal(target[:H * H * 2], torch.cat([s[:w_bytes] for s in new]))
assert torch.equal(target[H * H * 2:], new[0][w_bytes:])
print("%d values changed; payload %d bytes for %d weight bytes" % (sum(changed), size, plan.info.canonical_bytes))
