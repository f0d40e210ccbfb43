"""Helpers of the GPU parity tests: a device heap mirroring a host heap image
(tests/heap_image.py), so that a kernel's effect on the whole heap can be
compared byte for byte with the oracle's effect on the host image."""
from __future__ import annotations

import numpy as np
import torch


def device_heap(lay, host: np.ndarray, workspace_slots: int = 64):
    """A SymmetricHeap with the same partitions as ``lay`` holding ``host``
    (``workspace_slots`` 0: no load-balancing workspace, fixed shares)."""
    import gemm_gather_gb300 as gg
    sh = gg.SymmetricHeap(lay.H, lay.part_bytes, device="cuda", workspace_slots=workspace_slots)
    assert sh.part_bytes == lay.part_bytes
    sh.storage.copy_(torch.from_numpy(host).to("cuda"))
    return sh


def download(sh) -> np.ndarray:
    torch.cuda.synchronize()
    return sh.storage.cpu().numpy()


def first_diff(a: np.ndarray, b: np.ndarray, lay) -> str:
    idx = np.nonzero(a != b)[0]
    if len(idx) == 0:
        return "equal"
    i = int(idx[0])
    h, off = divmod(i, lay.part_bytes)
    return (f"{len(idx)} bytes differ; first at heap {h} offset {off} "
            f"(out_off {lay.out_off}, in_off {lay.in_off}): got {a[i]:#x} want {b[i]:#x}")
