"""A small decode loop as a serving engine drives libpagedattn.

Several sequences decode together for a number of steps, through a model of
a few layers (one KV cache per layer):
- pages come from the block allocator as sequences grow, and the
  sequences' block-table rows grow with them (pa_block_table_grow);
- each step makes one plan on the host (pa_plan_ex, with the early page
  copies of plan option early_kv), uploads it once, and every layer uses it:
  one launch per layer appends the step's token and attends
  (pa_append_decode_attention);
- halfway through, one sequence finishes: its pages are swapped out to
  pinned host memory (pa_copy_blocks) and given back to the allocator, and
  a new sequence takes its place in the batch.

torch tensors give the device memory and the stream; ``binding`` only
marshals arguments to the C ABI.  Run it on a GPU machine after building the
library:

    python -c "import __graft_entry__ as g; g.build()"
    python examples/serving_loop.py
"""

from __future__ import annotations

import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_kv_decode_24_gb300 import binding  # noqa: E402

PAGE = 16


def serve(prompt_lens=(90, 15, 300, 47), steps=24, layers=2, num_q_heads=8, num_kv_heads=2,
          head_dim=128, num_pages=160, seed=7):
    """Run the loop; returns what a caller needs to check the last step:
    dict(out=[per layer [B][Hq][D]], q=[per layer], k_pages=[...], v_pages=[...],
    block_table [B][max_pages], seq_lens [B], swapped=(host K, V of the finished
    sequence's pages, its page list, its K/V pages on the device before the
    swap), scale)."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D = len(prompt_lens), num_q_heads, num_kv_heads, head_dim
    max_pages = (max(prompt_lens) + steps + 2 * PAGE) // PAGE + 1
    shape = binding.make_shape(B, Hq, Hkv, D, PAGE, max_pages, num_pages)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    scale = D ** -0.5

    def rand(*s):
        return torch.from_numpy((rng.standard_normal(s) * 0.5).astype(np.float16)).to(dev)

    # One K and one V pool per layer.  Pages hold garbage until written.
    k_pages = [rand(num_pages, Hkv, PAGE, D) for _ in range(layers)]
    v_pages = [rand(num_pages, Hkv, PAGE, D) for _ in range(layers)]
    alloc = binding.BlockAllocator(num_pages)
    table = np.full((B, max_pages), -1, np.int32)
    lens = np.zeros(B, np.int32)
    # The prompts' pages (their K/V are the random pool contents: a prefill
    # would have written them).
    for b, L in enumerate(prompt_lens):
        alloc.grow(table[b], PAGE, 0, int(L))
        lens[b] = L
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = None
    swapped = None
    for step in range(steps):
        if step == steps // 2:
            # sequence 0 finishes: swap its pages out, free them, and start a
            # new sequence in its slot
            pages = table[0][table[0] >= 0].copy()
            host_k = torch.empty((len(pages), Hkv, PAGE, D), dtype=torch.float16).pin_memory()
            host_v = torch.empty_like(host_k).pin_memory()
            pairs = torch.from_numpy(np.stack([pages, np.arange(len(pages))], 1)
                                     .astype(np.int32)).to(dev)
            before = (k_pages[0][torch.from_numpy(pages).long().to(dev)].cpu(),
                      v_pages[0][torch.from_numpy(pages).long().to(dev)].cpu())
            binding.copy_blocks(host_k, k_pages[0], pairs, status)
            binding.copy_blocks(host_v, v_pages[0], pairs, status)
            torch.cuda.synchronize()
            swapped = (host_k, host_v, pages, before)
            alloc.free(pages)
            table[0] = -1
            lens[0] = 0
            alloc.grow(table[0], PAGE, 0, 20)   # the new sequence's 20-token prompt
            lens[0] = 20
        # every sequence decodes one token: grow its pages when it crosses one
        for b in range(B):
            alloc.grow(table[b], PAGE, int(lens[b]), int(lens[b]) + 1)
            lens[b] += 1
        bt_dev = torch.from_numpy(table).to(dev)
        sl_dev = torch.from_numpy(lens).to(dev)
        # host only.  early_kv: each layer's call reads its own layer's cache,
        # and seq_lens and the block table were copied in above, so a layer's
        # first page copies may start while the layer ahead still runs.
        plan = binding.Plan(shape, lens, sms, options=binding.plan_options(early_kv=1))
        if ws is None or ws.numel() < plan.workspace_bytes:
            ws = binding.alloc_workspace(plan, dev)
        binding.upload(plan, ws)                              # once per step
        outs, qs = [], []
        for layer in range(layers):
            q, k_new, v_new = rand(B, Hq, D), rand(B, Hkv, D), rand(B, Hkv, D)
            out = torch.empty_like(q)
            binding.append_decode(shape, plan, q, k_new, v_new, k_pages[layer], v_pages[layer],
                                  bt_dev, sl_dev, scale, out, ws, status)
            outs.append(out)
            qs.append(q)
        torch.cuda.synchronize()   # the plan's host buffer and ws are reused next step
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item()):#x}")
    return dict(out=outs, q=qs, k_pages=k_pages, v_pages=v_pages, block_table=table.copy(),
                seq_lens=lens.copy(), swapped=swapped, scale=scale, free=alloc.num_free())


if __name__ == "__main__":
    r = serve()
    print(f"{len(r['out'])} layers, last step's outputs {tuple(r['out'][0].shape)}, "
          f"sequence lengths {r['seq_lens'].tolist()}, {r['free']} pages free")
