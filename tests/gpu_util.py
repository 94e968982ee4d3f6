"""Helpers for the GPU tests: move synthetic workloads onto the device and
compare results with the oracle."""
import numpy as np
import torch

import synth

TOL = {"f16": 4e-3, "bf16": 1.6e-2}   # max |err| of attention outputs vs the fp64 oracle
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


def dev_bits(a: np.ndarray, dtype: str, device="cuda"):
    """uint16 bit patterns -> torch fp16/bf16 tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(TORCH_DTYPE[dtype]).to(device)


def host_bits(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class DevWorkload:
    """Device copies of a synth.Workload's inputs."""

    def __init__(self, w: synth.Workload, device="cuda"):
        self.w = w
        dt = w.dtype
        self.q = dev_bits(w.q, dt, device)
        self.k = dev_bits(w.k_cache, dt, device)
        self.v = dev_bits(w.v_cache, dt, device)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)
        self.out = torch.empty_like(self.q)
        self.k_new = None if w.k_new is None else dev_bits(w.k_new, dt, device)
        self.v_new = None if w.v_new is None else dev_bits(w.v_new, dt, device)
        self.slots = None if w.slot_mapping is None else torch.from_numpy(w.slot_mapping).to(device)
        self.pairs = (None if w.block_mapping is None or len(w.block_mapping) == 0
                      else torch.from_numpy(w.block_mapping).to(device))

    def step(self, pa, partition_size=0, workspace=None):
        """copy_blocks -> reshape_and_cache -> decode, as one decode step."""
        if self.pairs is not None:
            pa.copy_blocks(self.k, self.v, self.pairs)
        if self.slots is not None:
            pa.reshape_and_cache(self.k_new, self.v_new, self.k, self.v, self.slots)
        pa.decode(self.out, self.q, self.k, self.v, self.tables, self.lens, self.w.scale,
                  partition_size=partition_size, workspace=workspace)
        return self.out


def max_err(out, ref: np.ndarray) -> float:
    got = to_f64(out)
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.abs(got - ref).max()) if ref.size else 0.0
