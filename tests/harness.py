"""Harness-side expert models for the tests (not part of the method).

The pages leave expert computation to the caller (MORI-EP gfx1201 PR, Combine bullet: "expert
computation and applying routing weights to expert outputs remain the caller's responsibility").
The tests therefore model three experts, applied to the receive rows of whichever side
dispatched them (numpy for the oracle, torch on the GPU for the CUDA path), with the same IEEE
operation sequence on both so their outputs agree bit for bit:

* identity on a BF16 / FP16 payload: expert output = receive rows;
* identity on an FP8 payload: BF16 RNE of float(q) * scale[h // 128];
* per-expert scalar: for the receive row of rank r, y = BF16 RNE of the sequential FP32 sum over
  the token's experts e on rank r (top-k order) of (w_e * c_e) * x, no fused multiply-add.
"""
import numpy as np
import torch

FP8_BLOCK = 128


def _bf16_bits_to_f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32)


def _f32_to_bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def expert_np(wl, disp):
    """Expert output rows [W][W*M][H] (uint16 bits) computed on the CPU from receive rows."""
    if wl.dtype != "fp8" and wl.expert == "identity":
        return disp["recv_x"]
    W, M, H = wl.W, wl.M, wl.H
    out = np.zeros((W, W * M, H), dtype=np.uint16)
    for r in range(W):
        n = int(disp["recv_count"][r])
        if n == 0:
            continue
        if wl.dtype == "fp8":
            q = torch.from_numpy(np.ascontiguousarray(disp["recv_x"][r, :n])).view(torch.float8_e4m3fn)
            qf = q.to(torch.float32).numpy()
            sc = disp["recv_scales"][r, :n]
            y = qf * np.repeat(sc, FP8_BLOCK, axis=1)[:, :H]
            out[r, :n] = _f32_to_bf16_bits(y)
            continue
        X = _bf16_bits_to_f32(disp["recv_x"][r, :n])
        IDX = disp["recv_idx"][r, :n]
        Wt = disp["recv_w"][r, :n]
        c = wl.expert_scale
        acc = np.zeros((n, H), dtype=np.float32)
        for j in range(wl.k):
            m = (IDX[:, j] // wl.E) == r
            coef = (Wt[:, j] * c[IDX[:, j]]).astype(np.float32)
            term = coef[:, None] * X
            acc = np.where(m[:, None], acc + term, acc)
        out[r, :n] = _f32_to_bf16_bits(acc)
    return out


# e2m1 values of the 16 codes (sign in bit 3; code 8 is -0)
_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def mxfp4_dequant_np(q, sc):
    """Dequantising expert for MX FP4 receive rows: BF16 bits of e2m1(code) * 2^(c - 127) for
    q [..., H/2] packed codes and sc [..., H/32] e8m0 bytes.  Each product has at most two
    significant bits, so it and its BF16 value are exact."""
    H = q.shape[-1] * 2
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[:-1] + (H,))
    v = np.array(_E2M1, dtype=np.float32)[codes]
    bits = np.where(sc == 0, np.uint32(0x00400000), sc.astype(np.uint32) << np.uint32(23))
    scale = bits.astype(np.uint32).view(np.float32)
    return _f32_to_bf16_bits(v * np.repeat(scale, 32, axis=-1))


def mxfp4_dequant_torch(q, sc):
    """mxfp4_dequant_np with torch ops on the device: returns int16 BF16 bits [..., H]."""
    H = q.shape[-1] * 2
    codes = torch.stack([q & 0xF, q >> 4], dim=-1).reshape(*q.shape[:-1], H).long()
    v = torch.tensor(_E2M1, dtype=torch.float32, device=q.device)[codes]
    c = sc.to(torch.int32)
    bits = torch.where(c == 0, torch.full_like(c, 0x00400000), c << 23)
    scale = bits.view(torch.float32)
    return torch.mul(v, scale.repeat_interleave(32, dim=-1)).to(torch.bfloat16).view(torch.int16)


def expert_torch(wl, recv_x, recv_idx, recv_w, recv_scales, recv_count):
    """The same expert models on the GPU with torch ops (one op per IEEE step).

    Takes the device receive buffers (recv_x as a raw-bits tensor) and returns a device tensor
    [W][W*M][H] int16 of 16-bit result bits, or recv_x itself for the identity expert."""
    if wl.dtype != "fp8" and wl.expert == "identity":
        return recv_x
    W, M, H = wl.W, wl.M, wl.H
    dev = recv_x.device
    out = torch.zeros((W, W * M, H), dtype=torch.int16, device=dev)
    counts = recv_count.cpu().tolist()
    for r in range(W):
        n = int(counts[r])
        if n == 0:
            continue
        if wl.dtype == "fp8":
            qf = recv_x[r, :n].view(torch.float8_e4m3fn).to(torch.float32)
            sc = recv_scales[r, :n].repeat_interleave(FP8_BLOCK, dim=1)[:, :H]
            out[r, :n] = torch.mul(qf, sc).to(torch.bfloat16).view(torch.int16)
            continue
        X = recv_x[r, :n].view(torch.bfloat16).to(torch.float32)
        IDX = recv_idx[r, :n].long()
        Wt = recv_w[r, :n]
        c = torch.from_numpy(wl.expert_scale).to(dev)
        acc = torch.zeros((n, H), dtype=torch.float32, device=dev)
        for j in range(wl.k):
            m = torch.div(IDX[:, j], wl.E, rounding_mode="floor") == r
            coef = torch.mul(Wt[:, j], c[IDX[:, j]])
            term = torch.mul(coef[:, None], X)
            acc = torch.where(m[:, None], torch.add(acc, term), acc)
        out[r, :n] = acc.to(torch.bfloat16).view(torch.int16)
    return out
