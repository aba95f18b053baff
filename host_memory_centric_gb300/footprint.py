"""Device memory footprint of the training step as depth grows.

python -m host_memory_centric_gb300.footprint --config 14.7b --depths 12 24 [--device-ckpt]

For each depth, builds the model at that depth (full width), runs two
training steps and reports the device region the library carves, the peak of
device memory in use during the steps (cudaMemGetInfo, sampled around every
call) above the level before the model existed, and the host state.  With
host-resident checkpoints the carved region does not depend on depth.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import Model, configs, inputs


def used_bytes():
    free, total = torch.cuda.mem_get_info()
    return total - free


def measure(cfg_name: str, depth: int, ckpt_on_host: int) -> dict:
    c = configs.get(cfg_name, n_layers=depth)
    torch.cuda.synchronize()
    base = used_bytes()
    m = Model(c, seed=7, pin_store=1, ckpt_on_host=ckpt_on_host)
    peak = used_bytes() - base
    losses = []
    for s in range(2):
        m.set_tokens(inputs.tokens_for(c, s))
        losses.append(m.train_step(s))
        peak = max(peak, used_bytes() - base)
    m.sync()
    peak = max(peak, used_bytes() - base)
    st = m.stats()
    out = {"config": cfg_name, "n_layers": depth, "ckpt_on_host": ckpt_on_host,
           "device_region_GB": m.device_bytes / 1e9, "device_peak_used_GB": peak / 1e9,
           "host_store_GB": st["host_store_bytes"] / 1e9, "pinned_GB": st["pinned_bytes"] / 1e9,
           "params": sum(b["n_real"] for b in m.layout), "losses": losses}
    m.close()
    del m
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # hand the region back so the next depth starts from the same level
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="14.7b")
    ap.add_argument("--depths", type=int, nargs="+", default=[12, 24])
    ap.add_argument("--device-ckpt", action="store_true")
    a = ap.parse_args()
    for d in a.depths:
        print(json.dumps(measure(a.config, d, 0 if a.device_ckpt else 1)), flush=True)


if __name__ == "__main__":
    main()
