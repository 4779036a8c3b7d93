"""Device-memory plumbing around the C ABI: weight upload (bf16), workspaces, and the call
sequence of an n-block stack (embed -> blocks -> final).  No arithmetic happens here; every
step is one library call.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B

STREAMS = ("txt", "img")


def to_bf16(a, device="cuda") -> torch.Tensor:
    """A float32 array as a bf16 device tensor, rounded to nearest even (exact when the values are
    bf16-representable, as the seeded inputs are)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device=device).to(torch.bfloat16)


def to_f32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


class DeviceModel:
    """Weights of an n-block stack on the device.  `weights` has attributes dims, temb, embed,
    blocks (list of {stream: {name: array}}) and final, holding float32 arrays."""

    def __init__(self, weights, device="cuda"):
        self.dims = B.mf_dims(weights.dims.hidden, weights.dims.heads, weights.dims.channels,
                              weights.dims.mlp_ratio, weights.dims.freq_dim)
        up = lambda d: {k: to_bf16(v, device) for k, v in d.items()}        # noqa: E731
        self.temb = up(weights.temb)
        self.embed = up(weights.embed)
        self.blocks = [{s: up(b[s]) for s in STREAMS} for b in weights.blocks]
        self.final = up(weights.final)
        self.temb_struct = B.temb_struct(self.temb)
        self.block_structs = [B.block_struct(self.temb, b["txt"], b["img"]) for b in self.blocks]


class Workspace:
    """Device scratch sized for one plan: block forward, final layer and loss."""

    def __init__(self, plan, dims, device="cuda"):
        nb = max(B.mf_block_workspace_bytes(plan, dims), 256)
        nf = max(B.mf_final_workspace_bytes(plan, dims), 256)
        nl = max(B.mf_flow_loss_workspace_bytes(plan), 256)
        self.block = torch.empty(nb, dtype=torch.uint8, device=device)
        self.final = torch.empty(nf, dtype=torch.uint8, device=device)
        self.loss = torch.empty(nl, dtype=torch.uint8, device=device)


def run_stack(plan, model: DeviceModel, x_txt, zt_bf16, x_img, v, ws: Workspace, t=None,
              n_blocks=None, stream=None):
    """v = final(blocks(embed(z_t))) for the whole pack.  x_txt is updated in place; x_img is a
    [N_img][H] bf16 buffer the call overwrites; v is [N_img][C] f32."""
    d = model.dims
    B.mf_embed(plan, d, model.embed["w_in"], model.embed["b_in"], zt_bf16, x_img, stream=stream)
    # the first block leaves the timestep condition in the shared workspace; the rest reuse it
    for i, bs in enumerate(model.block_structs[:n_blocks]):
        B.mf_block_forward_ex(plan, d, bs, t, x_txt, x_img, ws.block, B.BLOCK_COND_GIVEN if i else 0,
                              stream=stream)
    f = model.final
    if model.block_structs[:n_blocks]:  # the blocks left the timestep condition in their workspace
        c = ws.block.data_ptr() + B.mf_block_workspace_layout(plan, d)[0]
        B.mf_final_ex(plan, d, model.temb_struct, f["w_fmod"], f["b_fmod"], f["w_out"], f["b_out"], t, x_img, v,
                      ws.final, c, stream=stream)
    else:
        B.mf_final(plan, d, model.temb_struct, f["w_fmod"], f["b_fmod"], f["w_out"], f["b_out"], t, x_img, v,
                   ws.final, stream=stream)
