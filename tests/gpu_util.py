"""Helpers shared by the GPU parity tests: move synthetic inputs to the device,
run the library through its Python binding, and build the oracle's own cache
from the same inputs (never from device results)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_paged_kv_q8_gb300 as k8

TOL = 2e-5          # |gpu - ref| <= TOL * max(1, |ref|), elementwise
CANARY = 0xA5


def dev_tensor(t, shape=None) -> torch.Tensor:
    """synth.Tensor -> CUDA tensor of its device dtype (bf16 bits or float32)."""
    if t.dtype == "bf16":
        x = torch.from_numpy(np.ascontiguousarray(t.dev).view(np.int16)).view(torch.bfloat16)
    else:
        x = torch.from_numpy(np.ascontiguousarray(t.f32))
    if shape is not None:
        x = x.reshape(shape)
    return x.cuda()


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref)))) if ref.size else 0.0


def make_caches(n_pages: int, P: int, H: int = 2, fmt: int = k8.FORMAT_K8V4):
    gpu = k8.PagedCache(n_pages, P, H, fmt)
    gpu.pages.fill_(CANARY)
    ref = oracle.Cache(n_pages, P, H, fmt, fill=CANARY)
    return gpu, ref


def append_both(gpu, ref, page_table: np.ndarray, pos: np.ndarray, k, v, chunk: int | None = None):
    """Append the same synthetic K/V ([n_seqs][n_tok][H][256]) on both sides."""
    pt_d = torch.from_numpy(np.ascontiguousarray(page_table, np.int32)).cuda()
    pos_d = torch.from_numpy(np.ascontiguousarray(pos, np.int64)).cuda()
    kd, vd = dev_tensor(k), dev_tensor(v)
    k8.kv_append_k8v4(gpu, pt_d, pos_d, kd, vd)
    ref.append(page_table, pos, k.f32, v.f32)
    return pt_d


def decode_gpu(gpu, q_dev: torch.Tensor, pt_d: torch.Tensor, lens: np.ndarray, max_len: int) -> np.ndarray:
    n = q_dev.shape[0]
    out = torch.empty(q_dev.shape, dtype=torch.float32, device="cuda")
    ws = k8.workspace(gpu, n, 1, max_len)
    k8.attn_k8v4_decode(gpu, q_dev, pt_d, torch.from_numpy(np.asarray(lens, np.int32)).cuda(), max_len, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def verify_gpu(gpu, q_dev: torch.Tensor, pt_d: torch.Tensor, steps: np.ndarray, max_len: int) -> np.ndarray:
    n, nq = q_dev.shape[0], q_dev.shape[1]
    out = torch.empty(q_dev.shape, dtype=torch.float32, device="cuda")
    ws = k8.workspace(gpu, n, nq, max_len)
    k8.attn_k8v4_verify(gpu, q_dev, pt_d, torch.from_numpy(np.asarray(steps, np.int32)).cuda(), max_len, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()
