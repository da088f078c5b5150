"""DeepSeekMoE layer forward on one B300 through the C ABI.

``MoELayer`` owns the (packed) weights and the per-batch buffers, all torch
device tensors, and runs one forward as four library calls on one stream:

    route -> permute -> expert_ffn -> combine   [-> update_bias]

h = u + sum_s FFN^(s)(u) + sum_i g_i FFN^(r)_i(u)
("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2, FFN-output equation),
with the auxiliary-loss-free bias step after the batch when asked.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional

import torch

from . import _lib


@dataclass
class Buffers:
    T: int
    topk_idx: torch.Tensor
    topk_gate: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    inv: torch.Tensor
    x_perm: torch.Tensor
    y_perm: torch.Tensor
    y_shared: Optional[torch.Tensor]
    h: torch.Tensor
    workspace: torch.Tensor
    # gate/up pre-activations of the last forward on this batch size when it
    # ran with save_for_backward (bf16 layers), for backward()
    act: Optional[torch.Tensor] = None
    act_shared: Optional[torch.Tensor] = None
    saved: bool = False


class MoELayer:
    def __init__(self, E: torch.Tensor, bias: torch.Tensor,
                 w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                 ws_gate: Optional[torch.Tensor] = None,
                 ws_up: Optional[torch.Tensor] = None,
                 ws_down: Optional[torch.Tensor] = None, top_k: int = 8,
                 h_dtype: torch.dtype = torch.float32, stream=None,
                 n_groups: int = 1, topk_groups: int = 1,
                 quant: Optional[str] = None, overlap_shared: bool = False):
        """quant="fp8": bf16 weights are quantized to e4m3 with block scales
        and the expert GEMMs run in e4m3 (activations and router stay
        bf16).  overlap_shared: run the shared experts on a side stream
        beside the permute (bf16 layers, T >= 1024, default stream only)."""
        if not E.is_cuda:
            raise ValueError("MoELayer needs CUDA tensors")
        if quant not in (None, "fp8"):
            raise ValueError(f"quant={quant!r}")
        if quant == "fp8" and E.dtype != torch.bfloat16:
            raise ValueError("fp8 layers take bf16 weights and activations")
        self.dtype = E.dtype
        self.code = "fp8" if quant == "fp8" else E.dtype
        self.N, self.d = E.shape
        self.I = w_gate.shape[1]
        self.S = 0 if ws_gate is None else ws_gate.shape[0]
        self.K = int(top_k)
        # group-limited routing when topk_groups < n_groups
        self.n_groups, self.topk_groups = int(n_groups), int(topk_groups)
        self.h_dtype = h_dtype
        # expert outputs: fp16 for bf16 and fp8 layers, fp32 for fp32 layers
        self.y_dtype = torch.float16 if E.dtype == torch.bfloat16 \
            else torch.float32
        self.E, self.bias = E, bias
        dev, dt = E.device, E.dtype
        if quant == "fp8":
            sh = self.shape(1)

            def buf(which):
                return torch.empty((_lib.fp8_weight_bytes(sh, which),),
                                   dtype=torch.uint8, device=dev)
            self.w_gu, self.w_down = buf(0), buf(1)
            self.ws_gu, self.ws_down = (buf(2), buf(3)) if self.S \
                else (None, None)
            _lib.pack_weights_fp8(sh, w_gate, w_up, w_down, ws_gate, ws_up,
                                  ws_down, self.w_gu, self.w_down, self.ws_gu,
                                  self.ws_down, stream)
        else:
            self.w_down = w_down
            self.w_gu = torch.empty((self.N, 2 * self.I, self.d), dtype=dt,
                                    device=dev)
            if self.S:
                self.ws_gu = torch.empty((2 * self.S * self.I, self.d),
                                         dtype=dt, device=dev)
                self.ws_down = torch.empty((self.d, self.S * self.I),
                                           dtype=dt, device=dev)
            else:
                self.ws_gu = self.ws_down = None
            _lib.pack_weights(self.shape(1), w_gate, w_up, ws_gate, ws_up,
                              ws_down, self.w_gu, self.ws_gu, self.ws_down,
                              stream)
        self._bufs: Dict[int, Buffers] = {}
        self._grads: Dict = {}
        self.overlap_shared = bool(overlap_shared)
        self._side = None

    def shape(self, T: int) -> _lib.MoeShape:
        return _lib.make_shape(T, self.d, self.N, self.K, self.S, self.I,
                               self.code)

    def _shared_side_stream(self, u: torch.Tensor):
        """Side stream for the shared experts when the overlap is on (bf16
        layers with shared experts and prefill-sized batches)."""
        if not (self.overlap_shared and self.S and self.code == self.dtype
                and self.dtype == torch.bfloat16 and u.shape[0] >= 1024):
            return None
        if self._side is None:
            self._side = torch.cuda.Stream(device=u.device)
        return self._side

    def buffers(self, T: int) -> Buffers:
        b = self._bufs.get(T)
        if b is not None:
            return b
        dev, dt, K = self.E.device, self.dtype, self.K
        A = T * K
        i32 = dict(dtype=torch.int32, device=dev)
        ws = _lib.workspace_size(self.shape(T))
        b = Buffers(
            T=T,
            topk_idx=torch.empty((T, K), **i32),
            topk_gate=torch.empty((T, K), dtype=torch.float32, device=dev),
            counts=torch.empty((self.N,), **i32),
            offsets=torch.empty((self.N + 1,), **i32),
            perm=torch.empty((max(A, 1),), **i32),
            inv=torch.empty((T, K), **i32),
            x_perm=(torch.empty((max(_lib.x_perm_bytes(self.shape(T)), 256),),
                                dtype=torch.uint8, device=dev)
                    if self.code == "fp8"
                    else torch.empty((max(A, 1), self.d), dtype=dt,
                                     device=dev)),
            y_perm=torch.empty((max(A, 1), self.d), dtype=self.y_dtype,
                               device=dev),
            y_shared=(torch.empty((T, self.d), dtype=self.y_dtype,
                                  device=dev) if self.S else None),
            h=torch.empty((T, self.d), dtype=self.h_dtype, device=dev),
            workspace=torch.empty((max(ws, 256),), dtype=torch.uint8,
                                  device=dev),
        )
        self._bufs[T] = b
        return b

    def forward(self, u: torch.Tensor, update_bias: bool = False,
                gamma: float = 1e-3, stream=None,
                out: Optional[torch.Tensor] = None,
                save_for_backward: bool = False) -> torch.Tensor:
        """h for u[T, d]; the result lives in this layer's buffer for T, or
        in ``out`` ([T, d], the layer's output dtype) when given.  With
        ``save_for_backward`` (bf16 layers) the expert FFNs also store their
        gate/up pre-activations, and the next backward() on this batch uses
        them instead of recomputing them."""
        T = u.shape[0]
        b = self.buffers(T)
        sh = self.shape(T)
        if save_for_backward:
            if self.code != torch.bfloat16:
                raise ValueError("save_for_backward: bf16 layers only")
            if b.act is None:
                dev = self.E.device
                b.act = torch.empty((max(T * self.K, 1), 2 * self.I),
                                    dtype=torch.float16, device=dev)
                b.act_shared = (torch.empty((T, 2 * self.S * self.I),
                                            dtype=torch.float16, device=dev)
                                if self.S else None)
        b.saved = False
        _lib.route_grouped(sh, self.n_groups, self.topk_groups, u, self.E,
                           self.bias, b.topk_idx, b.topk_gate, b.counts,
                           b.workspace, stream)
        side = (self._shared_side_stream(u)
                if stream is None and not save_for_backward else None)
        if side is not None:
            # the shared experts need no routing: they run on a side stream
            # beside the permute and join before the routed experts' output
            # is combined
            main = torch.cuda.current_stream(u.device)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                _lib.expert_ffn_part(sh, 2, None, None, None, None, u,
                                     self.ws_gu, self.ws_down, None,
                                     b.y_shared, b.workspace)
        _lib.permute(sh, u, b.topk_idx, b.counts, b.offsets, b.perm, b.inv,
                     b.x_perm, b.workspace, stream)
        if side is not None:
            _lib.expert_ffn_part(sh, 1, b.x_perm, b.offsets, self.w_gu,
                                 self.w_down, u, None, None, b.y_perm, None,
                                 b.workspace)
            main.wait_stream(side)
        elif save_for_backward:
            _lib.expert_ffn_train(sh, b.x_perm, b.offsets, self.w_gu,
                                  self.w_down, u, self.ws_gu, self.ws_down,
                                  b.y_perm, b.y_shared, b.act, b.act_shared,
                                  b.workspace, stream)
            b.saved = True
        else:
            _lib.expert_ffn(sh, b.x_perm, b.offsets, self.w_gu, self.w_down,
                            u, self.ws_gu, self.ws_down, b.y_perm, b.y_shared,
                            b.workspace, stream)
        h = b.h if out is None else out
        if h.shape != b.h.shape or h.dtype != b.h.dtype or h.device != u.device:
            raise ValueError("out must match the layer's output buffer")
        _lib.combine(sh, u, b.y_perm, b.y_shared, b.inv, b.topk_gate, h,
                     stream)
        if update_bias:
            _lib.update_bias(self.N, b.counts, T * self.K, gamma, self.bias,
                             stream)
        return h

    __call__ = forward

    def backward(self, u: torch.Tensor, dh: torch.Tensor,
                 grad_dtype: torch.dtype = torch.float32, stream=None):
        """Gradients of the layer for the upstream gradient dh [T, d] (bf16),
        after a forward on the same u (its routing, slots and expert outputs
        are reused, and its gate/up pre-activations when it ran with
        save_for_backward).  Returns a dict: du [T, d] and dE [N, d] fp32; dw_gate,
        dw_up [N, I, d], dw_down [N, d, I] and, with shared experts, dws_gate,
        dws_up [S, I, d], dws_down [S, d, I] as grad_dtype.  The tensors are
        this layer's buffers for (T, grad_dtype), overwritten by the next
        call.  bf16 layers only; the bias gets no gradient (it only selects).
        """
        if self.code != torch.bfloat16:
            raise ValueError("backward: bf16 layers only")
        T = u.shape[0]
        if T not in self._bufs:
            raise ValueError("backward: run the forward on this batch first")
        b = self._bufs[T]
        sh = self.shape(T)
        key = (T, grad_dtype)
        g = self._grads.get(key)
        if g is None:
            dev, N, d, I, S = self.E.device, self.N, self.d, self.I, self.S
            f32 = dict(dtype=torch.float32, device=dev)
            gd = dict(dtype=grad_dtype, device=dev)
            g = dict(du=torch.empty((T, d), **f32),
                     dE=torch.empty((N, d), **f32),
                     dw_gate=torch.empty((N, I, d), **gd),
                     dw_up=torch.empty((N, I, d), **gd),
                     dw_down=torch.empty((N, d, I), **gd))
            if S:
                g.update(dws_gate=torch.empty((S, I, d), **gd),
                         dws_up=torch.empty((S, I, d), **gd),
                         dws_down=torch.empty((S, d, I), **gd))
            ws = torch.empty((_lib.backward_workspace_size(sh) + 256,),
                             dtype=torch.uint8, device=dev)
            off = (-ws.data_ptr()) % 256
            g["_ws"] = ws[off:]
            self._grads[key] = g
        _lib.backward(sh, dh, u, self.E, b.topk_idx, b.topk_gate, b.offsets,
                      b.inv, b.y_perm, self.w_gu, self.w_down, self.ws_gu,
                      self.ws_down, g["du"], g["dE"], g["dw_gate"],
                      g["dw_up"], g["dw_down"], g.get("dws_gate"),
                      g.get("dws_up"), g.get("dws_down"), g["_ws"], stream,
                      act=b.act if b.saved else None,
                      act_shared=b.act_shared if b.saved else None)
        return {k: v for k, v in g.items() if not k.startswith("_")}

    def forward_host(self, u_host, h_host, update_bias: bool = False,
                     gamma: float = 1e-3) -> None:
        """Run the layer on a sequence of host batches: ``u_host[i]`` (pinned
        CPU tensors [T, d], the layer's input dtype) -> ``h_host[i]`` (pinned
        CPU tensors [T, d], the output dtype).  Batch i+1 is uploaded and
        batch i-1 read back on copy streams while batch i computes: two
        device input and two device output buffers, ordered by events.
        Returns once every result is on the host.  With ``update_bias`` each
        batch is a training step (the bias moves after each batch, in batch
        order)."""
        n = len(u_host)
        if n == 0:
            return
        dev = self.E.device
        T = u_host[0].shape[0]
        for x, y in zip(u_host, h_host):
            if x.shape[0] != T or y.shape[0] != T:
                raise ValueError("all batches must have the same T")
        b = self.buffers(T)
        comp = torch.cuda.current_stream(dev)
        up = torch.cuda.Stream(device=dev)
        down = torch.cuda.Stream(device=dev)
        u_dev = [torch.empty((T, self.d), dtype=self.dtype, device=dev)
                 for _ in range(2)]
        h_dev = [torch.empty_like(b.h) for _ in range(2)]
        uploaded = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]   # u buffer free
        computed = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]  # h buffer free
        for e in consumed + read_back:
            e.record(comp)

        def upload(i):
            j = i % 2
            up.wait_event(consumed[j])
            with torch.cuda.stream(up):
                u_dev[j].copy_(u_host[i], non_blocking=True)
                uploaded[j].record(up)

        upload(0)
        for i in range(n):
            j = i % 2
            if i + 1 < n:
                upload(i + 1)
            comp.wait_event(uploaded[j])
            comp.wait_event(read_back[j])
            self.forward(u_dev[j], update_bias=update_bias, gamma=gamma,
                         out=h_dev[j])
            consumed[j].record(comp)
            computed[j].record(comp)
            down.wait_event(computed[j])
            with torch.cuda.stream(down):
                h_host[i].copy_(h_dev[j], non_blocking=True)
                read_back[j].record(down)
        down.synchronize()
        # the caller's stream sees every step's writes (bias, buffers)
        comp.wait_stream(down)

    def graph(self, u: torch.Tensor, update_bias: bool = False,
              gamma: float = 1e-3, dh: Optional[torch.Tensor] = None,
              grad_dtype: torch.dtype = torch.float32):
        """Capture one forward on ``u`` (a fixed device buffer) into a CUDA
        graph and return a function that replays it.  Every call of the step
        is asynchronous with no host synchronisation, so the whole step --
        route, permute, expert FFNs, combine (and the bias update when asked)
        -- replays as one graph launch.  Write new tokens into ``u`` between
        replays; the result is this layer's buffer for ``u.shape[0]``.  With
        ``update_bias`` every replay moves the bias once.  With ``dh`` (a
        fixed device buffer of upstream gradients) the backward pass is
        captured after the forward (which, for bf16 layers, saves its gate/up
        pre-activations for it), and a replay returns (h, gradients) -- one
        training step per graph launch."""
        T = u.shape[0]
        self.buffers(T)
        side = torch.cuda.Stream(device=u.device)
        side.wait_stream(torch.cuda.current_stream(u.device))
        train = dh is not None and self.code == torch.bfloat16
        with torch.cuda.stream(side):      # first-use set-up outside capture
            self.forward(u, save_for_backward=train)
            if dh is not None:
                self.backward(u, dh, grad_dtype=grad_dtype)
        torch.cuda.current_stream(u.device).wait_stream(side)
        torch.cuda.synchronize(u.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            h = self.forward(u, update_bias=update_bias, gamma=gamma,
                             save_for_backward=train)
            grads = (self.backward(u, dh, grad_dtype=grad_dtype)
                     if dh is not None else None)

        def replay():
            g.replay()
            return h if grads is None else (h, grads)
        replay.graph = g
        return replay

    # --- checkpoint of the routing bias (the layer's only changing state) --
    def save_state(self, path: str, step: int) -> None:
        """Write the current bias and the index of the next step."""
        from .checkpoint import save_bias
        torch.cuda.current_stream().synchronize()
        save_bias(path, self.bias, step)

    def load_state(self, path: str) -> int:
        """Restore the bias in place; returns the step to resume at."""
        from .checkpoint import load_bias
        b, step = load_bias(path)
        if b.size != self.N:
            raise ValueError(f"checkpoint has {b.size} experts, layer {self.N}")
        self.bias.copy_(torch.from_numpy(b))
        return step
