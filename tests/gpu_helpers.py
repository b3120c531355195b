"""Shared helpers of the GPU parity tests: move seeded host inputs to the device in their
declared dtype, run the library, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import sub_byte_quantized_gb300 as kvq
from oracle import attention as OA

ATOL, RTOL = 2e-3, 1e-3        # |gpu - oracle| <= ATOL + RTOL * |oracle|


def to_device(arr_f32: np.ndarray, bits: np.ndarray | None, dtype: str, dev="cuda") -> torch.Tensor:
    """The exact device tensor of an input: bf16/f16 from their bits, f32 as is."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)
    if dtype == "f16":
        return torch.from_numpy(np.ascontiguousarray(arr_f32).astype(np.float16)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(arr_f32, dtype=np.float32)).to(dev)


def device_inputs(inp: dict, dev="cuda") -> dict:
    return {n: to_device(inp[n], inp.get(n + "_bits"), inp["dtype"], dev) for n in ("q", "k", "v")}


def fill_both(w, inp: dict, capacity: int | None = None, dev="cuda", fill: int | None = None):
    """Store the workload's K/V into a device cache and an oracle cache the same way:
    a bulk store of the first `fill` tokens, then the rest as a second append."""
    B, H, S, D = inp["k"].shape
    cap = capacity or S
    dcache = kvq.KVCache(w.layout, B, H, D, cap, n_recent=w.n_recent, device=dev)
    ocache = OA.OracleCache(w.layout, B, H, D, cap, n_recent=w.n_recent)
    d = device_inputs(inp, dev)
    n_fill = min(S, w.n_fill if fill is None else fill)
    for lo, hi in ((0, n_fill), (n_fill, S)):
        if hi > lo:
            kvq.store(dcache, d["k"][:, :, lo:hi].contiguous(), d["v"][:, :, lo:hi].contiguous(), lo)
            ocache.store(inp["k"][:, :, lo:hi], inp["v"][:, :, lo:hi], lo)
    return dcache, ocache, d


def planes_equal(dcache, ocache, kv_len: int | None = None) -> None:
    """Bit-exact comparison of every stored plane (tokens [0, kv_len))."""
    n = kv_len or dcache.capacity
    for t in ("k", "v"):
        dp, op = dcache.planes[t], ocache.planes[t]
        got = dp["payload"][:, :, :n].cpu().numpy()
        want = op["payload"][:, :, :n]
        if not np.array_equal(got, want):
            idx = np.argwhere(got != want)[0]
            raise AssertionError(f"{t} payload differs first at {tuple(idx)}: {got[tuple(idx)]} vs {want[tuple(idx)]}")
        gs = dp["scale"][:, :, :n].cpu().numpy()
        ws = op["scale"][:, :, :n]
        assert np.array_equal(gs.view(np.uint16 if gs.dtype == np.float16 else np.uint32),
                              ws.view(np.uint16 if ws.dtype == np.float16 else np.uint32)), f"{t} scale differs"
        if "zero" in op:
            assert np.array_equal(dp["zero"][:, :, :n].cpu().numpy().view(np.uint16),
                                  op["zero"][:, :, :n].view(np.uint16)), f"{t} zero differs"
        if "ring" in op:
            assert np.array_equal(dp["recent"].cpu().numpy().view(np.uint32), op["ring"].view(np.uint32)), \
                f"{t} window differs"


def check_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    tol = ATOL + RTOL * np.abs(ref)
    bad = err > tol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {i}: "
                             f"got {got[i]!r} want {ref[i]!r}; max ratio {np.max(err / tol):.3f}")
    return {"max_abs": float(err.max()), "max_ratio": float((err / tol).max())}
