"""A DeepSeekMoE FP8 layer held in device memory, driven through the C ABI.

MoELayer owns the layer's device tensors (centroids, bias, E4M3 weight
stacks and their 128x128 block scales), a workspace, and the output
buffers of one forward pass.  Quantising the float32 master weights and the
whole forward run in libmoefp8's kernels; torch only allocates memory.
"""
from __future__ import annotations

import torch

from . import lib, workloads


class MoELayer:
    def __init__(self, d: int, E: int, K: int, S: int, I: int, device="cuda"):
        self.d, self.E, self.K, self.S, self.I = d, E, K, S, I
        self.G = E + S
        dev = torch.device(device)
        self.device = dev
        self.centroids = torch.zeros((E, d), dtype=torch.float32, device=dev)
        self.bias = torch.zeros((E,), dtype=torch.float32, device=dev)
        self.w_gate = torch.zeros((self.G, I, d), dtype=torch.uint8, device=dev)
        self.w_up = torch.zeros((self.G, I, d), dtype=torch.uint8, device=dev)
        self.w_down = torch.zeros((self.G, d, I), dtype=torch.uint8, device=dev)
        self.s_gate = torch.ones((self.G, I // 128, d // 128), dtype=torch.float32, device=dev)
        self.s_up = torch.ones((self.G, I // 128, d // 128), dtype=torch.float32, device=dev)
        self.s_down = torch.ones((self.G, d // 128, I // 128), dtype=torch.float32, device=dev)
        self._ws = None
        self._T_ws = -1
        # group-limited routing (moe_route_grouped); 0 groups: plain top-K
        self.n_groups = self.topk_groups = self.group_topk = 0

    def set_group_routing(self, n_groups: int, topk_groups: int, group_topk: int):
        self.n_groups, self.topk_groups, self.group_topk = n_groups, topk_groups, group_topk

    # ------------------------------------------------------------ set-up
    @classmethod
    def from_config(cls, cfg: workloads.LayerConfig, device="cuda", gen_device=None) -> "MoELayer":
        """Synthetic layer of a workload: seeded centroids, bias and master
        weights, each weight matrix quantised 128x128 by moe_quant_128x128.
        gen_device: where the generator draws the numbers (default: the
        layer's device; "cpu" gives the same bits and launches no generator
        kernels on the GPU, only the quantiser's)."""
        L = cls(cfg.d, cfg.E, cfg.K, cfg.S, cfg.I, device)
        gdev = L.device if gen_device is None else torch.device(gen_device)
        L.set_group_routing(cfg.n_groups, cfg.topk_groups, cfg.group_topk)
        L.centroids.copy_(workloads.centroids(cfg, gdev))
        L.bias.copy_(workloads.bias(cfg, gdev))
        for g in range(L.G):
            for which, q, s in (("gate", L.w_gate, L.s_gate), ("up", L.w_up, L.s_up),
                                ("down", L.w_down, L.s_down)):
                w = workloads.master_weight(cfg, which, g, gdev).to(L.device)
                lib.moe_quant_128x128(w, q[g], s[g])
        return L

    def set_group(self, g: int, gate, up, down):
        """Install already-quantised (codes, scales) pairs for group g."""
        for (q, s), dq, ds in ((gate, self.w_gate, self.s_gate), (up, self.w_up, self.s_up),
                               (down, self.w_down, self.s_down)):
            dq[g].copy_(torch.as_tensor(q))
            ds[g].copy_(torch.as_tensor(s))

    def struct(self) -> lib.moe_layer_t:
        return lib.moe_layer_t(self.d, self.E, self.K, self.S, self.I,
                               self.centroids.data_ptr(), self.bias.data_ptr(),
                               self.w_gate.data_ptr(), self.w_up.data_ptr(),
                               self.w_down.data_ptr(), self.s_gate.data_ptr(),
                               self.s_up.data_ptr(), self.s_down.data_ptr(),
                               self.n_groups, self.topk_groups, self.group_topk)

    def workspace(self, T: int) -> torch.Tensor:
        if self._ws is None or self._T_ws < T:
            n = lib.moe_workspace_size(self.struct(), T)
            self._ws = torch.empty(n + 256, dtype=torch.uint8, device=self.device)
            self._T_ws = T
        return self._ws

    def outputs(self, T: int) -> dict:
        dev = self.device
        return {"h": torch.empty((T, self.d), dtype=torch.float32, device=dev),
                "idx": torch.empty((T, self.K), dtype=torch.int32, device=dev),
                "gate": torch.empty((T, self.K), dtype=torch.float32, device=dev),
                "counts": torch.empty((self.E,), dtype=torch.int32, device=dev),
                "tie": torch.empty((T,), dtype=torch.uint8, device=dev)}

    # ----------------------------------------------------------- forward
    def forward(self, u: torch.Tensor, out: dict | None = None, stream=None) -> dict:
        T = u.shape[0]
        out = self.outputs(T) if out is None else out
        return lib.moe_forward(self.struct(), u, self.workspace(T), out, stream)

    def forward_host(self, u_host: list, h_host: list, gamma: float = 0.0, streams=None) -> list:
        """The layer over batches that live in pinned host memory, pipelined
        (moe_forward_host): batch k+1's upload and batch k-1's download overlap
        batch k's compute; with gamma != 0 the bias steps after every batch.
        Returns the two device buffer sets (the last two batches' routing).
        Asynchronous on the three streams (created here unless given)."""
        T = u_host[0].shape[0] if u_host else 0
        if streams is None:
            streams = getattr(self, "_host_streams", None)
            if streams is None:
                streams = self._host_streams = (torch.cuda.Stream(self.device),
                                                torch.cuda.Stream(self.device),
                                                torch.cuda.Stream(self.device))
        bufs = getattr(self, "_host_bufs", None)
        if bufs is None or bufs[0]["u"].shape[0] != T:
            bufs = self._host_bufs = [dict(self.outputs(T),
                                           u=torch.empty((T, self.d), dtype=torch.bfloat16,
                                                         device=self.device)) for _ in range(2)]
        # the streams start after everything already queued on the current one
        cur = torch.cuda.current_stream(self.device)
        for s in streams:
            s.wait_stream(cur)
        lib.moe_forward_host(self.struct(), T, u_host, h_host, gamma, bufs, self.workspace(T),
                             *streams)
        return bufs

    def forward_pipelined(self, us: list, gamma: float = 0.0, reserve_sms: int = 0,
                          outs: list | None = None, streams=None) -> list:
        """The layer over device-resident batches with two micro-batches in
        flight (moe_forward_pipelined): batch k's routing and dispatch, and
        batch k-1's combine, run on a side stream while the expert GEMMs of the
        other batch run on the GEMM stream (their grids leave reserve_sms SMs
        free).  With gamma != 0 the bias steps after every batch.  Returns the
        per-batch output dicts; asynchronous on the two streams (the current
        stream is made to wait for them)."""
        if not us:
            return []
        T = us[0].shape[0]
        outs = [dict(self.outputs(T), u=u) for u in us] if outs is None else outs
        if getattr(self, "_ws2", None) is None or self._ws2.numel() < self.workspace(T).numel():
            self._ws2 = torch.empty_like(self.workspace(T))
        if streams is None:
            streams = getattr(self, "_pipe_streams", None)
            if streams is None:
                streams = self._pipe_streams = (torch.cuda.Stream(self.device),
                                                torch.cuda.Stream(self.device))
        cur = torch.cuda.current_stream(self.device)
        for s in streams:
            s.wait_stream(cur)
        lib.moe_forward_pipelined(self.struct(), outs, gamma, self.workspace(T), self._ws2,
                                  reserve_sms, *streams)
        for s in streams:
            cur.wait_stream(s)
        return outs

    def pipelined_status(self, stream=None) -> int:
        """Device status of the two workspaces of forward_pipelined (syncs)."""
        a = self.status(stream)
        ws = getattr(self, "_ws2", None)
        b = lib.moe_check_device_status(ws[:16].view(torch.int32), stream) if ws is not None else 0
        return a or b

    def capture_forward(self, u: torch.Tensor, out: dict | None = None):
        """A CUDA graph of moe_forward on the fixed buffers u and out (decode
        steps: the launches of one forward become one graph launch).  Refill u
        in place and call .replay(); out holds the results.  Returns
        (graph, out)."""
        T = u.shape[0]
        out = self.outputs(T) if out is None else out
        ws = self.workspace(T)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            for _ in range(2):                       # first-call set-up outside the capture
                lib.moe_forward(self.struct(), u, ws, out, side)
        torch.cuda.current_stream(self.device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            lib.moe_forward(self.struct(), u, ws, out, side)
        return g, out

    # ---------------------------------------------------------- backward
    def prepare_backward(self, stream=None):
        """Transposed weight blocks for the input gradient (after every change
        of the weights)."""
        dev, G, d, I = self.device, self.G, self.d, self.I
        if getattr(self, "_bwd_w", None) is None:
            self._bwd_w = (torch.empty((G, I, d), dtype=torch.uint8, device=dev),
                           torch.empty((G, I // 128, d // 128), dtype=torch.float32, device=dev),
                           torch.empty((G, d, 2 * I), dtype=torch.uint8, device=dev),
                           torch.empty((G, d // 128, 2 * I // 128), dtype=torch.float32, device=dev))
        lib.moe_prepare_backward_weights(self.struct(), *self._bwd_w, stream)

    def backward_dgrad(self, u: torch.Tensor, dh: torch.Tensor, fwd: dict, stream=None) -> torch.Tensor:
        """du of the forward that just ran on u (fwd: its outputs; the layer's
        workspace still holds its dispatch state)."""
        if getattr(self, "_bwd_w", None) is None:
            self.prepare_backward(stream)
        T = u.shape[0]
        n = lib.moe_backward_workspace_size(self.struct(), T)
        if getattr(self, "_bwd_ws", None) is None or self._bwd_ws.numel() < n:
            self._bwd_ws = torch.empty(n + 256, dtype=torch.uint8, device=self.device)
        B = lib.moe_layer_bwd_t(*(t.data_ptr() for t in self._bwd_w))
        return lib.moe_backward_dgrad(self.struct(), B, u, dh, fwd, self.workspace(T), self._bwd_ws,
                                      stream=stream)

    def backward_wgrad(self, T: int, out: tuple | None = None, stream=None) -> tuple:
        """Weight gradients (dW_gate [G, I, d], dW_up [G, I, d], dW_down [G, d, I],
        float32) of the batch of T tokens whose forward and backward_dgrad just
        ran; out: optional preallocated triple."""
        if getattr(self, "_bwd_ws", None) is None:
            raise RuntimeError("backward_wgrad needs the workspace of backward_dgrad")
        n = lib.moe_wgrad_workspace_size(self.struct(), T)
        if getattr(self, "_wg_ws", None) is None or self._wg_ws.numel() < n:
            self._wg_ws = torch.empty(n + 256, dtype=torch.uint8, device=self.device)
        G, d, I = self.G, self.d, self.I
        if out is None:
            out = (torch.empty((G, I, d), dtype=torch.float32, device=self.device),
                   torch.empty((G, I, d), dtype=torch.float32, device=self.device),
                   torch.empty((G, d, I), dtype=torch.float32, device=self.device))
        lib.moe_backward_wgrad(self.struct(), T, self.workspace(T), self._bwd_ws, self._wg_ws, *out,
                               stream=stream)
        return out

    def backward_status(self, stream=None) -> int:
        ws = getattr(self, "_bwd_ws", None)
        return lib.moe_check_device_status(ws[:16].view(torch.int32), stream) if ws is not None else 0

    def update_bias(self, counts: torch.Tensor, T: int, gamma: float, stream=None):
        lib.moe_update_bias(counts, self.bias, T, self.K, gamma, stream)

    def status(self, stream=None) -> int:
        """Reads and clears the device status word of the last forward (syncs)."""
        ws = self._ws
        return lib.moe_check_device_status(ws[:16].view(torch.int32), stream) if ws is not None else 0
