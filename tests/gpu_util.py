"""Helpers shared by the GPU tests: upload of host-generated inputs, the
tolerance check, and oracle evaluation on sampled rows."""
from __future__ import annotations

import numpy as np

import oracle
import synth

REL_L2 = 1e-5          # relative L2 error bound on every product
ABS_PER_SQRT_K = 1e-3  # max |err| <= 1e-3 * sqrt(K) * max half-scale of the matrix


def torch():
    import torch as _t
    return _t


def act_dtype(act):
    t = torch()
    return t.float16 if act == synth.ACT_F16 else t.bfloat16


def upload_w(Wh: np.ndarray):
    return torch().from_numpy(np.ascontiguousarray(Wh).reshape(-1)).cuda()


def upload_x(bits: np.ndarray, act: int):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(act_dtype(act))


def max_halfscale(Wh: np.ndarray, variant: int) -> float:
    bb = synth.block_bytes(variant)
    sc = Wh.reshape(-1, bb)[:, 16:].ravel()
    return max(oracle.halfscale(int(s)) for s in np.unique(sc))


def assert_close(Y, Yref: np.ndarray, K: int, max_hs: float, what: str = ""):
    Y = np.asarray(Y, dtype=np.float64)
    assert Y.shape == Yref.shape, (Y.shape, Yref.shape)
    assert np.all(np.isfinite(Y)), f"{what}: non-finite outputs"
    err = Y - Yref
    nref = np.linalg.norm(Yref)
    rel = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    amax = np.max(np.abs(err)) if err.size else 0.0
    bound = ABS_PER_SQRT_K * np.sqrt(K) * max_hs
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert amax <= bound, f"{what}: max abs err {amax:.3e} > {bound:.3e}"
    return rel, amax
