"""One decode step of one layer through libpagedattn from Python.

torch tensors give the device memory and the stream; ``binding`` only
marshals arguments to the C ABI (include/pagedattn.h).  Run it on a GPU
machine after building the library:

    python -c "import __graft_entry__ as g; g.build()"
    python examples/decode_step.py
"""

from __future__ import annotations

import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_kv_decode_24_gb300 import binding  # noqa: E402


def decode_step(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, num_sms=None):
    """Append the new token's K/V rows and attend, in one kernel launch.

    q [B][Hq][D] and k_new, v_new [B][Hkv][D] (fp16 or bf16); pools
    k_pages, v_pages [P][Hkv][16][D]; block_table [B][max_pages] int32 (-1
    pad); seq_lens [B] int32 counting the new token; all on the GPU.
    Returns (out [B][Hq][D], status), status a device int32 holding PA_DEV_*
    bits (0 when all went well) once the stream is synchronised.
    """
    shape = binding.shape_of(q, k_pages, block_table)
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    plan = binding.Plan(shape, seq_lens.cpu().numpy(), num_sms)   # host only
    ws = binding.alloc_workspace(plan, q.device)                  # one per call in flight
    binding.upload(plan, ws)                                      # once per plan
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    out = torch.empty_like(q)
    binding.append_decode(shape, plan, q, k_new, v_new, k_pages, v_pages, block_table, seq_lens,
                          q.shape[-1] ** -0.5, out, ws, status)
    # One uploaded plan serves every layer of a step; make a new plan when
    # seq_lens change.
    return out, status


if __name__ == "__main__":
    from paged_kv_decode_24_gb300 import workloads
    w = workloads.make_custom(seq_lens=[300, 37, 1025], num_q_heads=8, num_kv_heads=2,
                              head_dim=128, seed=91)
    dev = lambda a: torch.from_numpy(a).cuda()
    out, status = decode_step(dev(w.q), dev(w.k_new), dev(w.v_new), dev(w.k_pages),
                              dev(w.v_pages), dev(w.block_table), dev(w.seq_lens))
    torch.cuda.synchronize()
    print(f"out {tuple(out.shape)} {out.dtype}, status {int(status.item()):#x}")
