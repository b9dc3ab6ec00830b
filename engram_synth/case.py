"""All random inputs of one workload, drawn on a device.

Table sizes (rows per layer) come from the caller, who derives them from the
layout; nothing here computes the layout or any step of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import gen


@dataclass
class Case:
    w: object
    batch: dict                       # numpy: input_ids, cu_seqlens, sequence_ids, token_mask, lookback_ids, token_map
    tables: list                      # per layer: {"fmt", "table", "scales", "num_rows"} (device tensors)
    wkv: list                         # per layer: bf16 [N, K]
    q_weight: list                    # per layer: bf16 [hc, H]
    k_weight: list
    streams: list                     # per layer: fp32 [T, hc, H] (initial values)
    extra: dict = field(default_factory=dict)


def layer_formats(w) -> tuple:
    """Table format of each layer: ``w.extra["layer_formats"]`` if given, else ``w.table_format``."""
    fmts = tuple(w.extra.get("layer_formats", (w.table_format,) * w.layers))
    if len(fmts) != w.layers:
        raise ValueError(f"{w.name}: {len(fmts)} layer formats for {w.layers} layers")
    return fmts


def make_tables(w, rows_per_layer, device, seed: int):
    out = []
    for layer, (rows, fmt) in enumerate(zip(rows_per_layer, layer_formats(w))):
        s = seed * 100 + layer
        rows = int(rows)
        if fmt == "fp8":
            t, sc = gen.fp8_table(rows, w.head_dim, w.table_std, s, device)
        elif fmt == "q2k":
            t, sc = gen.q2k_table(rows, s, device), None
        elif fmt == "bf16":
            t, sc = gen.bf16_table(rows, w.head_dim, w.table_std, s, device), None
        else:
            raise ValueError(fmt)
        out.append({"fmt": fmt, "table": t, "scales": sc, "num_rows": rows})
    return out


def make_case(w, rows_per_layer, device="cpu", seed: int | None = None, with_tables: bool = True,
              with_weights: bool = True) -> Case:
    """with_weights False leaves out wkv, the gate weights and the streams (for looking at the
    hash or the gather alone)."""
    seed = w.seed if seed is None else seed
    batch = gen.batch_inputs(w, seed)
    T = w.tokens
    tables = make_tables(w, rows_per_layer, device, seed) if with_tables else []
    wkv, qs, ks, st = [], [], [], []
    for layer in range(w.layers if with_weights else 0):
        s = seed * 100 + layer
        wkv.append(gen.wkv_weight(w.N, w.K, w.wkv_std, s, device))
        q, k = gen.gate_weights(w.hc, w.hidden, w.qk_std, s, device)
        qs.append(q)
        ks.append(k)
        st.append(gen.streams(T, w.hc, w.hidden, s, device))
    return Case(w, batch, tables, wkv, qs, ks, st)


def to_device(a, device, dtype=None):
    """numpy array (or None) -> contiguous tensor on device."""
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)
