"""Checkpoint of the layer's only state that changes during training: the
routing bias b[N_r] (float32) and the step index.

The bias moves by the auxiliary-loss-free rule after every step
("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2), so resuming a run at
step k needs exactly the bias after step k-1.  The file holds it as raw
float32 so that a resumed run is bit-identical to an uninterrupted one.

Format (little-endian): 8-byte magic ``MOEBIAS1``, uint32 N, int64 step,
then N float32 values.  Writes go to a temporary file first and are renamed
into place, so a crash never leaves a torn checkpoint.
"""
from __future__ import annotations

import os
import struct
from typing import Tuple

import numpy as np

MAGIC = b"MOEBIAS1"
_HEAD = struct.Struct("<8sIq")


def save_bias(path: str, bias, step: int) -> None:
    """Write ``bias`` (a torch tensor on any device, or a numpy array) and
    the index of the next step to run."""
    if hasattr(bias, "detach"):
        arr = bias.detach().to("cpu").numpy()
    else:
        arr = np.asarray(bias)
    if arr.dtype != np.float32 or arr.ndim != 1:
        raise ValueError("bias must be a 1-D float32 vector")
    tmp = f"{path}.tmp{os.getpid()}"
    with open(tmp, "wb") as f:
        f.write(_HEAD.pack(MAGIC, arr.size, int(step)))
        f.write(arr.astype("<f4").tobytes())
        f.flush()
        os.fsync(f.fileno())
    os.replace(tmp, path)


def load_bias(path: str) -> Tuple[np.ndarray, int]:
    """Read a checkpoint; returns (bias float32 [N], step)."""
    with open(path, "rb") as f:
        head = f.read(_HEAD.size)
        if len(head) != _HEAD.size:
            raise ValueError(f"{path}: truncated header")
        magic, n, step = _HEAD.unpack(head)
        if magic != MAGIC:
            raise ValueError(f"{path}: not a bias checkpoint")
        body = f.read()
    if len(body) != 4 * n:
        raise ValueError(f"{path}: expected {n} values, found "
                         f"{len(body) / 4:g}")
    return np.frombuffer(body, dtype="<f4").astype(np.float32), int(step)
