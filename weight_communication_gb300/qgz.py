"""One qgZ reduce step over R simulated ranks, composed from the C-ABI calls.

ZeROPlusPlus.md §1.2 (quantized gradient communication): each rank
block-quantizes its gradient to int4, an all-to-all replaces the
reduce-scatter, and the receivers reduce in full precision -- flat, or
intra-group first and inter-group second.  "Merge LoCo with Zero++" (DeepSpeed
PR #6730), Overview: the gradient is compensated with the rank's
error-feedback buffer before quantization, at the cost of that buffer's
memory and no extra time.

`QgzReducer` owns the device buffers of one problem (error feedback, send
buffers, first-hop buffers, reduced shards) and runs a step as 2 launches
(flat) or 3 launches (hierarchical) on one stream, or, with `fused=True`, as
1 launch (flat: wc_qgz_step_fused and its bf16/int8-buffer forms) or 2
(hierarchical: wc_qgz_first_hop_fused and its forms, then the second hop),
bit for bit the same.  `DevicePipeline` overlaps
each step's reduce with the next quantization, `HostPipeline` runs steps from
and to host memory with the copies overlapped, and `GraphedStep` replays a
step captured in a CUDA graph.
"""
from __future__ import annotations

import torch

from . import binding


class QgzReducer:
    """Device state and launches of one (R, N, G, B) quantized reduce.

    error feedback : fp32 or bf16 [R, N], or int8 [R, N] with fp32 scales
                     [R, N/B]; persistent across steps (zeroed at start)
    codes, scales  : int4 send buffers [R, N/2] bytes and [R, N/B] fp32
    hop1 codes/sc. : first-hop outputs [G*N/2], [G*N/B] (G > 1 only)
    out            : reduced shards [N] (= [R][S]), fp32 or bf16
    """

    def __init__(self, N: int, R: int, G: int = 1, B: int = 256, err_scale: float = 1.0,
                 err_beta: float = 0.0, use_ef: bool = True, out_dtype=torch.float32,
                 out_scale: float = 1.0, device="cuda", ef_dtype=torch.float32,
                 hop1_ef: bool = False, fused: bool = False):
        """ef_dtype: torch.float32, torch.bfloat16 for the half-size error
        buffer (wc_ef_quant_int4_bf16ef), or torch.int8 for the quarter-size
        one (wc_ef_quant_int4_int8ef: int8 codes in self.ef, one fp32 scale per
        block in self.ef_scales).  hop1_ef (G > 1): keep an fp32 error
        for the first hop's requantization too (wc_dequant_reduce_requant_ef),
        with the same err_scale and err_beta.  fused: step() quantizes and
        reduces (flat) or quantizes and runs the first hop, with its error
        buffer if any (hierarchical), in one kernel, still writing the send
        buffers; it takes every error buffer form, and B >= 128."""
        self.N, self.R, self.G, self.B = N, R, G, B
        self.err_scale, self.err_beta = err_scale, err_beta
        self.out_scale = out_scale
        self.device = torch.device(device)
        dev = self.device
        if ef_dtype not in (torch.float32, torch.bfloat16, torch.int8):
            raise TypeError("ef_dtype must be float32, bfloat16 or int8")
        self.ef = torch.zeros(R * N, dtype=ef_dtype, device=dev) if use_ef else None
        self.ef_scales = (torch.zeros(R * N // B, dtype=torch.float32, device=dev)
                          if use_ef and ef_dtype == torch.int8 else None)
        self.codes = torch.empty(R * N // 2, dtype=torch.uint8, device=dev)
        self.scales = torch.empty(R * N // B, dtype=torch.float32, device=dev)
        if G > 1:
            self.codes1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
            self.scales1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
        else:
            self.codes1 = self.scales1 = None
        self.ef1 = torch.zeros(G * N, dtype=torch.float32, device=dev) if (hop1_ef and G > 1) else None
        self.out = torch.empty(N, dtype=out_dtype, device=dev)
        if fused:
            if B < 128:
                raise ValueError(f"fused steps need B >= 128 (one warp per block), got B={B}")
        self.fused = fused

    @property
    def launches_per_step(self) -> int:
        if self.fused:
            return 2 if self.G > 1 else 1
        return 3 if self.G > 1 else 2

    def quantize(self, g: torch.Tensor, stream=None, send=None) -> None:
        """EF-quant of every rank into the send buffers (self.codes,
        self.scales, or the (codes, scales) pair `send`)."""
        codes, scales = send if send is not None else (self.codes, self.scales)
        if self.ef is not None and self.ef.dtype == torch.bfloat16:
            binding.ef_quant_int4_bf16ef(g.reshape(-1), self.ef, codes, scales, self.N,
                                         self.R, self.G, self.B, self.err_scale, self.err_beta,
                                         stream)
        elif self.ef is not None and self.ef.dtype == torch.int8:
            binding.ef_quant_int4_int8ef(g.reshape(-1), self.ef, self.ef_scales, codes, scales,
                                         self.N, self.R, self.G, self.B, self.err_scale,
                                         self.err_beta, stream)
        else:
            binding.ef_quant_int4(g.reshape(-1), self.ef, codes, scales, self.N, self.R,
                                  self.G, self.B, self.err_scale, self.err_beta, stream)

    def reduce_first_hop(self, stream=None, send=None) -> None:
        """G > 1: the intra-group dequant-reduce-requant into codes1/scales1."""
        codes, scales = send if send is not None else (self.codes, self.scales)
        if self.ef1 is not None:
            binding.dequant_reduce_requant_ef(codes, scales, self.codes1, self.scales1,
                                              self.ef1, self.N, self.R, self.G, self.B,
                                              self.err_scale, self.err_beta, stream)
        else:
            binding.dequant_reduce_requant(codes, scales, self.codes1, self.scales1,
                                           self.N, self.R, self.G, self.B, stream)

    def reduce_last_hop(self, stream=None, out: torch.Tensor | None = None,
                        send=None) -> torch.Tensor:
        """The dequant-reduce into the shards (self.out unless `out` is
        given): flat, or the inter-group hop."""
        out = self.out if out is None else out
        if self.G > 1:
            binding.dequant_reduce(self.codes1, self.scales1, out, self.N, self.R, self.G,
                                   self.B, self.out_scale, stream)
        else:
            codes, scales = send if send is not None else (self.codes, self.scales)
            binding.dequant_reduce(codes, scales, out, self.N, self.R, 1, self.B,
                                   self.out_scale, stream)
        return out

    def reduce(self, stream=None) -> torch.Tensor:
        if self.G > 1:
            self.reduce_first_hop(stream)
        return self.reduce_last_hop(stream)

    def step(self, g: torch.Tensor, stream=None, out: torch.Tensor | None = None) -> torch.Tensor:
        """Quantize every rank's gradient g ([R, N] bf16 on the device) and
        reduce; returns the [N] reduced shards (destination-major), in
        self.out unless `out` is given."""
        if self.fused:
            return self.step_fused(g, stream, out)
        self.quantize(g, stream)
        if self.G > 1:
            self.reduce_first_hop(stream)
        return self.reduce_last_hop(stream, out=out)

    def step_fused(self, g: torch.Tensor, stream=None,
                   out: torch.Tensor | None = None) -> torch.Tensor:
        """The step in the fused kernels: flat, one launch that quantizes every
        rank and reduces every shard; hierarchical, one launch that quantizes
        every rank and runs the first hop (with its error buffer, if the
        reducer keeps one), then the second hop."""
        out = self.out if out is None else out
        if self.G > 1:
            binding.qgz_first_hop_fused(g.reshape(-1), self.ef, self.codes, self.scales,
                                        self.codes1, self.scales1, self.N, self.R, self.G,
                                        self.B, self.err_scale, self.err_beta, stream,
                                        ef1=self.ef1, ef_scales=self.ef_scales)
            return self.reduce_last_hop(stream, out=out)
        binding.qgz_step_fused(g.reshape(-1), self.ef, self.codes, self.scales, out, self.N,
                               self.R, self.B, self.err_scale, self.err_beta, self.out_scale,
                               stream, ef_scales=self.ef_scales)
        return out

    def step_host(self, g_host: torch.Tensor, g_dev: torch.Tensor, out_host: torch.Tensor,
                  stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """End-to-end step from host memory: copy g_host (pinned, [R, N] bf16)
        into g_dev, run the step, copy the shards into out_host (pinned), all
        on one stream; the caller synchronizes."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            g_dev.copy_(g_host, non_blocking=True)
            self.step(g_dev, s)
            out_host.copy_(self.out, non_blocking=True)
        return out_host


class DevicePipeline:
    """Back-to-back steps with each step's reduce on a second stream, beside
    the next step's EF-quant.

    The quantization is HBM-bound and the reduce issue-bound, so running them
    side by side lets the reduce hide under the quantization.  Ordering uses
    events between the two streams, never a host wait (the llm.c ZeRO-2
    review asks the same of its NCCL stream).  Two send buffers rotate:
    step i quantizes into send[i % 2] once step i-2's reduce has read it.
    The error buffer sees the steps in order (one quantization stream); so
    does the first-hop error and the output (one reduce stream).
    """

    def __init__(self, red: QgzReducer):
        if red.fused:
            raise ValueError("a fused step has no separate reduce to overlap; "
                             "use QgzReducer.step or HostPipeline")
        self.red = red
        self.send = [(red.codes, red.scales),
                     (torch.empty_like(red.codes), torch.empty_like(red.scales))]
        self.quant_stream = torch.cuda.Stream(red.device)
        # the reduce's blocks go ahead of the quantization's pending ones, so
        # the two kernels actually share the GPU instead of queueing
        self.reduce_stream = torch.cuda.Stream(red.device, priority=-1)
        self.quantized = [torch.cuda.Event() for _ in range(2)]
        self.reduced = [torch.cuda.Event() for _ in range(2)]
        self.count = 0
        self.timer = None      # optional callable(kind, i, "begin"|"end", stream)

    def step(self, g: torch.Tensor) -> torch.Tensor:
        """Enqueue one step; returns red.out, valid once reduce_stream has run
        the step (wait on it, or synchronize)."""
        red, i = self.red, self.count
        b = i % 2
        qs, rs = self.quant_stream, self.reduce_stream
        if i >= 2:
            qs.wait_event(self.reduced[b])
        if self.timer:
            self.timer("quant", i, "begin", qs)
        red.quantize(g, qs, send=self.send[b])
        if self.timer:
            self.timer("quant", i, "end", qs)
        self.quantized[b].record(qs)
        rs.wait_event(self.quantized[b])
        if self.timer:
            self.timer("reduce", i, "begin", rs)
        if red.G > 1:
            red.reduce_first_hop(rs, send=self.send[b])
        red.reduce_last_hop(rs, send=self.send[b])
        if self.timer:
            self.timer("reduce", i, "end", rs)
        self.reduced[b].record(rs)
        self.count += 1
        return red.out


class HostPipeline:
    """Steps of a QgzReducer from pinned host gradients to pinned host shards,
    with each step's host->device copy, kernels and device->host copy
    overlapped with its neighbours' on three streams (the two copy
    directions use separate copy engines; the kernels keep their order on
    one stream, so the error buffer sees the steps in sequence).

    Two device buffers of each kind rotate: step i's gradient goes to
    g_dev[i % 2] once step i-2's quantization has read it, and its shards
    come from out_dev[i % 2] once step i-2's copy to the host has finished.
    """

    def __init__(self, red: QgzReducer):
        self.red = red
        dev = red.device
        self.g_dev = [torch.empty(red.R * red.N, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.out_dev = [torch.empty_like(red.out) for _ in range(2)]
        self.h2d = torch.cuda.Stream(dev)
        self.comp = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.g_loaded = [torch.cuda.Event() for _ in range(2)]
        self.g_consumed = [torch.cuda.Event() for _ in range(2)]
        self.out_ready = [torch.cuda.Event() for _ in range(2)]
        self.out_copied = [torch.cuda.Event() for _ in range(2)]
        self._started = [False, False]

    def run(self, g_host: list, out_host: list) -> None:
        """Step i reads g_host[i] (pinned, R*N bf16) and writes out_host[i]
        (pinned, like red.out).  Asynchronous: the caller synchronizes (or
        waits on self.d2h) before reading out_host."""
        red = self.red
        for i, (gh, oh) in enumerate(zip(g_host, out_host)):
            b = i % 2
            with torch.cuda.stream(self.h2d):
                if self._started[b]:
                    self.h2d.wait_event(self.g_consumed[b])
                self.g_dev[b].copy_(gh.view(-1), non_blocking=True)
                self.g_loaded[b].record(self.h2d)
            with torch.cuda.stream(self.comp):
                self.comp.wait_event(self.g_loaded[b])
                if red.fused:
                    # the fused launch writes the shards while it reads g
                    if self._started[b]:
                        self.comp.wait_event(self.out_copied[b])
                    red.step_fused(self.g_dev[b], self.comp, out=self.out_dev[b])
                    self.g_consumed[b].record(self.comp)
                else:
                    red.quantize(self.g_dev[b], self.comp)
                    self.g_consumed[b].record(self.comp)
                    if self._started[b]:
                        self.comp.wait_event(self.out_copied[b])
                    if red.G > 1:
                        red.reduce_first_hop(self.comp)
                    red.reduce_last_hop(self.comp, out=self.out_dev[b])
                self.out_ready[b].record(self.comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.out_ready[b])
                oh.copy_(self.out_dev[b], non_blocking=True)
                self.out_copied[b].record(self.d2h)
            self._started[b] = True


class GraphedStep:
    """One QgzReducer step captured in a CUDA graph: replay() issues its one
    to three kernels with a single graph launch, which takes the host's
    per-call work (argument checks, marshalling, one launch per kernel) off
    the step.  That matters when the step is short: a small problem is
    bound by how fast the host can launch, not by the GPU.

    The graph reads its gradient from one fixed device buffer, `g`: copy each
    step's gradient there (in stream order) before replay().  The error
    buffers, the send buffers and `red.out` are the reducer's own, so replays
    advance the error feedback exactly as step() calls do.  The caller keeps
    the reducer's buffers alive while the graph exists.
    """

    def __init__(self, red: QgzReducer, stream: torch.cuda.Stream | None = None):
        self.red = red
        dev = red.device
        self.g = torch.zeros(red.R * red.N, dtype=torch.bfloat16, device=dev)
        self.stream = stream if stream is not None else torch.cuda.Stream(dev)
        self.graph = torch.cuda.CUDAGraph()
        self.stream.wait_stream(torch.cuda.current_stream(dev))
        # the capture records the launches without running them, so the
        # reducer's state is untouched until the first replay
        with torch.cuda.graph(self.graph, stream=self.stream):
            red.step(self.g, self.stream)

    def replay(self) -> torch.Tensor:
        """Run one step on the contents of self.g; returns red.out (valid in
        stream order after the replay)."""
        self.graph.replay()
        return self.red.out
