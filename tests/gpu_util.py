"""Helpers for the GPU parity tests: device copies, bit comparison, guard bands."""
import hashlib
import os
from contextlib import contextmanager

import numpy as np

GUARD = 64  # floats of sentinel before and after every output buffer
SENTINEL = np.uint32(0x7FBADBAD)


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def sha(a) -> str:
    return hashlib.sha256(bits(a).tobytes()).hexdigest()


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded_output(init: np.ndarray):
    """A device buffer holding ``init`` between two sentinel guard bands.
    Returns (buffer, view) where view is the part the kernel may write."""
    import torch
    flat = np.empty(init.size + 2 * GUARD, np.float32)
    flat.view(np.uint32)[:] = SENTINEL
    flat[GUARD:GUARD + init.size] = init.reshape(-1)
    buf = torch.from_numpy(flat).cuda()
    return buf, buf[GUARD:GUARD + init.size]


def guards_intact(buf) -> bool:
    h = bits(buf.cpu().numpy())
    return bool((h[:GUARD] == SENTINEL).all() and (h[-GUARD:] == SENTINEL).all())


@contextmanager
def forced_config(var: str, cfg):
    old = os.environ.get(var)
    if cfg is None:
        os.environ.pop(var, None)
    else:
        os.environ[var] = str(cfg)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop(var, None)
        else:
            os.environ[var] = old


def assert_bits_equal(got, want, what=""):
    g, w = bits(got), bits(want)
    if not np.array_equal(g, w):
        bad = np.argwhere(g != w)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} outputs differ; first at {i}: "
                             f"got {g[i]:#010x} want {w[i]:#010x}")
