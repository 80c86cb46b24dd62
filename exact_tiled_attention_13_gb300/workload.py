"""Put one of the synthetic attention workloads on the GPU and launch the forward pass.

    python -m exact_tiled_attention_13_gb300.workload --workload 3 --iters 3

generates the seeded inputs of the workload, copies them to cuda:0, launches
the forward pass `--iters` times on the current stream and synchronises. It is the command
the profiler summaries under profiles/ were taken with.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


class DeviceWorkload:
    """Seeded host inputs (pinned) and device buffers of one synthetic workload."""

    def __init__(self, workload_id: int, device="cuda"):
        import torch

        import synth

        self.id = workload_id
        self.w = synth.WORKLOADS[workload_id]
        self.host = synth.make_inputs(self.w, workload_id)
        w = self.w

        def pinned(arr, dtype):
            t = torch.from_numpy(np.ascontiguousarray(arr))
            if dtype is not None:
                t = t.view(dtype)
            return t.pin_memory()

        self.Q_h = pinned(self.host["Q"].view(np.int16), torch.bfloat16)
        self.K_h = pinned(self.host["K"].view(np.int16), torch.bfloat16)
        self.V_h = pinned(self.host["V"].view(np.int16), torch.bfloat16)
        self.C_h = None if self.host["C"] is None else pinned(self.host["C"], None)
        self.ck_h = None if self.host.get("ckey") is None else pinned(self.host["ckey"], None)
        self.Q = self.Q_h.to(device)
        self.K = self.K_h.to(device)
        self.V = self.V_h.to(device)
        self.C = None if self.C_h is None else self.C_h.to(device)
        self.ckey = None if self.ck_h is None else self.ck_h.to(device)
        self.workspace = None
        self.launches_per_step = 1
        if w.split_kv:
            import exact_tiled_attention_13_gb300 as eta

            self.workspace = eta.splitkv_workspace(w.mode, w.BH, w.N, w.Nkv, w.d, w.dv, 0,
                                                   device=device)
            self.launches_per_step = 1 if self.workspace is None else 2
        odt = torch.float32 if w.out_dtype == "f32" else torch.bfloat16
        self.O = torch.empty(w.BH, w.N, w.dv, dtype=odt, device=device)
        self.LSE = torch.empty(w.BH, w.N, dtype=torch.float32, device=device)
        self.O_h = torch.empty(self.O.shape, dtype=odt).pin_memory()
        self.LSE_h = torch.empty(self.LSE.shape, dtype=torch.float32).pin_memory()
        # The plain forward pass streams host tensors through attn_fwd_host end to end.
        self.staging = None
        if not w.split_kv and not w.backward:
            import exact_tiled_attention_13_gb300 as eta

            self.staging = eta.host_staging(w.mode, w.BH, w.N, w.Nkv, w.d, w.dv,
                                            1 if w.out_dtype == "f32" else 0, device=device)
        if w.backward:
            import exact_tiled_attention_13_gb300 as eta

            # The forward pass once, for O and LSE; the step is the backward pass.
            eta.attn_fwd_ex(self.Q, self.K, self.V, w.mode, self.C, self.ckey, w.scale, self.O,
                            self.LSE)
            self.O_h.copy_(self.O)
            self.LSE_h.copy_(self.LSE)
            self.dO_h = pinned(self.host["dO"].view(np.int16), torch.bfloat16)
            self.dO = self.dO_h.to(device)
            self.dQ = torch.empty(w.BH, w.N, w.d, dtype=torch.float32, device=device)
            self.dK = torch.empty(w.BH, w.Nkv, w.d, dtype=torch.float32, device=device)
            self.dV = torch.empty(w.BH, w.Nkv, w.dv, dtype=torch.float32, device=device)
            self.grads_h = [torch.empty(t.shape, dtype=torch.float32).pin_memory()
                            for t in (self.dQ, self.dK, self.dV)]
            self.workspace = eta.bwd_workspace(w.BH, w.N, device=device)
            self.launches_per_step = 3
            # End to end the backward pass streams host tensors through attn_bwd_host.
            self.bwd_staging = eta.bwd_host_staging(w.mode, w.BH, w.N, w.Nkv, w.d, w.dv,
                                                    1 if w.out_dtype == "f32" else 0, device=device)

    def launch(self, stream=None):
        import exact_tiled_attention_13_gb300 as eta

        if self.w.backward:
            eta.attn_bwd(self.Q, self.K, self.V, self.O, self.dO, self.LSE, self.w.mode, self.C,
                         self.ckey, self.w.scale, self.dQ, self.dK, self.dV, self.workspace,
                         stream=stream)
        elif self.w.split_kv:
            eta.attn_fwd_splitkv(self.Q, self.K, self.V, self.w.mode, self.C, self.ckey,
                                 self.w.scale, self.O, self.LSE, workspace=self.workspace,
                                 stream=stream)
        else:
            eta.attn_fwd_ex(self.Q, self.K, self.V, self.w.mode, self.C, self.ckey, self.w.scale,
                            self.O, self.LSE, stream=stream)

    def _inputs(self):
        pairs = [(self.Q, self.Q_h), (self.K, self.K_h), (self.V, self.V_h), (self.C, self.C_h),
                 (self.ckey, self.ck_h)]
        if self.w.backward:
            pairs += [(self.O, self.O_h), (self.LSE, self.LSE_h), (self.dO, self.dO_h)]
        return [(d, h) for d, h in pairs if d is not None]

    def _outputs(self):
        if self.w.backward:
            return list(zip((self.dQ, self.dK, self.dV), self.grads_h))
        return [(self.O, self.O_h), (self.LSE, self.LSE_h)]

    def h2d_bytes(self) -> int:
        return sum(h.numel() * h.element_size() for _, h in self._inputs())

    def d2h_bytes(self) -> int:
        return sum(d.numel() * d.element_size() for d, _ in self._outputs())

    def end_to_end(self, stream):
        """One call the way a host-side user makes it: pinned host inputs in, host outputs out.
        The plain forward and the backward pass are one attn_fwd_host / attn_bwd_host call
        (uploads, kernels and downloads of chunks of heads overlapped); the split pass copies,
        launches and copies back."""
        import exact_tiled_attention_13_gb300 as eta

        w = self.w
        if self.staging is not None:
            eta.attn_fwd_host(self.Q_h, self.K_h, self.V_h, w.mode, self.C_h, self.ck_h, w.scale,
                              self.O_h, self.LSE_h, self.staging, stream=stream)
            return
        if w.backward:
            eta.attn_bwd_host(self.Q_h, self.K_h, self.V_h, self.O_h, self.dO_h, self.LSE_h, w.mode,
                              self.C_h, self.ck_h, w.scale, *self.grads_h, self.bwd_staging,
                              stream=stream)
            return
        for d, h in self._inputs():
            d.copy_(h, non_blocking=True)
        self.launch(stream)
        for d, h in self._outputs():
            h.copy_(d, non_blocking=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3, 4, 5, 6, 7, 8])
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    import torch

    wl = DeviceWorkload(args.workload)
    for _ in range(args.iters):
        wl.launch()
    torch.cuda.synchronize()
    import exact_tiled_attention_13_gb300 as eta

    code, word = eta.attn_device_status(None)
    if code != eta.ATTN_OK:
        raise SystemExit(f"watchdog tripped: {word:#x}")
    print(f"workload {args.workload} ({wl.w.name}): {args.iters} launches done")


if __name__ == "__main__":
    main()
