"""Run a few steps of one workload of the 8B-like layer, for a profiler.

  python -m mamba_ssm_layer_gb300.profile_case decode_b1  [--steps 4]
  python -m mamba_ssm_layer_gb300.profile_case decode_b64 [--steps 3]
  python -m mamba_ssm_layer_gb300.profile_case prefill_1k [--steps 2]
  python -m mamba_ssm_layer_gb300.profile_case prefill_1k_w8a8 [--steps 2]

Small on purpose: at most a few hundred MB on the device, with the weights
rotated over two copies so that a decode step's inputs are not left in L2 by
the step before.  The library must have been built (``__graft_entry__.build``).
"""
from __future__ import annotations

import argparse
import copy

import torch

from . import abi, synth
from .layer import DeviceLayer, to_dev


def _copy_layer(dl: DeviceLayer) -> DeviceLayer:
    new = copy.copy(dl)
    new.t = {k: (None if v is None else v.clone()) for k, v in dl.t.items()}
    t, d = new.t, dl.dims_dict
    new.struct = abi.M2Layer(
        t["norm_w"].data_ptr(),
        abi.weight_struct(t["in_w"], t["in_s"], dl.n_in, d["hidden"], dl.struct.in_proj.fmt),
        t["conv_w"].data_ptr(), t["conv_b"].data_ptr(), t["A_log"].data_ptr(), t["D"].data_ptr(),
        t["dt_bias"].data_ptr(), t["gnorm_w"].data_ptr(),
        abi.weight_struct(t["out_w"], t["out_s"], d["hidden"], dl.d_inner, dl.struct.out_proj.fmt))
    return new


def main() -> None:
    p = argparse.ArgumentParser()
    p.add_argument("workload", choices=["decode_b1", "decode_b64", "prefill_1k", "prefill_1k_w8a8"])
    p.add_argument("--steps", type=int, default=4)
    a = p.parse_args()
    abi.lib()
    d = synth.NEMOTRON_H_8B
    if a.workload.startswith("prefill_1k"):
        T = 1024
        dl = DeviceLayer(synth.make_layer(d, synth.WL_8B_PREFILL_1K))
        ws = dl.workspace_varlen(1, T)
        st = dl.new_state(1)
        x = to_dev(synth.make_hidden(T, d["hidden"], synth.WL_8B_PREFILL_1K, 0, 0))
        for _ in range(a.steps):
            dl.prefill_varlen(x, [0, T], (st[0][:1], st[1][:1], st[2][:1]), ws,
                              w8a8=a.workload.endswith("w8a8"))
    else:
        B = 1 if a.workload == "decode_b1" else 64
        wl = synth.WL_8B_DECODE_B1 if B == 1 else synth.WL_8B_DECODE_B64
        base = DeviceLayer(synth.make_layer(d, wl))
        reps = [base, _copy_layer(base)]
        sts = [r.new_state(B) for r in reps]
        ws = base.workspace(B, 0)
        x = to_dev(synth.make_hidden(B, d["hidden"], wl, 0, 0))
        for i in range(a.steps):  # each step hints the other replica, as the decode benchmark does
            reps[i % 2].decode(x, sts[i % 2], ws, ahead=reps[(i + 1) % 2] if B == 1 else None)
    torch.cuda.synchronize()
    st = abi.m2_device_status()
    if st != abi.M2_OK:
        raise SystemExit(f"device status {st}")
    print(f"{a.workload}: {a.steps} steps, {abi.m2_launch_count()} launches")


if __name__ == "__main__":
    main()
