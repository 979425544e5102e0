"""Random-weight decode loop: the LM head's share of a decode step.

FlashSampling's end-to-end claim is about time per output token: fusing the
sampler into the LM head shortens every decode step of a serving engine
(summary page, "Results", second paragraph; arXiv abstract).  This module
measures that share on its own terms, without a serving engine, trained
weights or datasets: a decoder body with the Llama-3-8B layer shapes and
random bf16 weights runs one step per token, then the LM head samples the next
token -- with the fused sampler (``fs_sample``) or with the unfused pipeline
(``fs_sample_unfused``: logits to HBM, softmax, sample) -- and the sampled ids
are embedded (tied to the LM-head matrix) as the next step's input.

The body is a stand-in for the weight traffic and GEMMs of a decoder layer:
RMSNorm, the q/k/v/o projections (no attention mixing: there is no KV cache
here, so its reads, which depend on the context length, are left out) and the
SwiGLU MLP.  Its kernels are PyTorch's (cuBLAS GEMMs, elementwise); only the
LM head and the sampling run this library's kernels.  The embedding and body
of a step are one CUDA-graph replay, so the step is bound by the GPU, not by
the host's launch rate.  Timing: CUDA events on one stream, around the whole
loop for the step time and around each step's LM-head call for the head time
(see ``DecodeLoop.run``).
"""

from dataclasses import dataclass

from . import binding as fs

# Llama-3-8B decoder shapes (hidden, q heads x head dim, kv width, MLP width).
LLAMA3_8B_LAYER = dict(d=4096, q=4096, kv=1024, ffn=14336)


@dataclass
class StepTiming:
    step_us: float          # whole decode step
    head_us: float          # LM head + sampling (the library's launch(es))

    @property
    def share(self):
        return self.head_us / self.step_us


class DecodeLoop:
    """A random-weight decoder body plus the LM head W [V, d] (bf16, device).

    ``layers`` decoder layers of the shapes in ``layer`` (default: Llama-3-8B),
    weights ~ N(0, 1/fan_in) in bf16, drawn on the device from ``seed``.
    """

    def __init__(self, W, layers=32, layer=None, seed=0):
        import torch
        self.torch = torch
        self.W = W
        V, d = W.shape
        shape = dict(LLAMA3_8B_LAYER if layer is None else layer)
        assert shape["d"] == d, "the body's hidden size must match the LM head's"
        g = torch.Generator(device=W.device).manual_seed(seed)

        def mat(n_in, n_out):
            m = torch.randn((n_out, n_in), generator=g, device=W.device, dtype=torch.float32)
            return (m * (n_in ** -0.5)).to(torch.bfloat16)

        self.layers = []
        for _ in range(layers):
            self.layers.append(dict(
                qkv=mat(d, shape["q"] + 2 * shape["kv"]), o=mat(shape["q"], d),
                gate_up=mat(d, 2 * shape["ffn"]), down=mat(shape["ffn"], d)))
        self.q = shape["q"]
        self.ffn = shape["ffn"]

    @staticmethod
    def _rms(x):
        xf = x.float()
        return (xf * (xf.pow(2).mean(-1, keepdim=True) + 1e-6).rsqrt()).to(x.dtype)

    def body(self, x):
        """The decoder layers on hidden states x [B, d] (bf16)."""
        torch = self.torch
        for L in self.layers:
            y = self._rms(x) @ L["qkv"].t()
            x = x + y[:, : self.q] @ L["o"].t()             # projections only (no KV cache)
            gu = self._rms(x) @ L["gate_up"].t()
            g, u = gu[:, : self.ffn], gu[:, self.ffn:]
            x = x + (torch.nn.functional.silu(g) * u) @ L["down"].t()
        return self._rms(x)

    def _head(self, x, temp, seed, step, ids, mx, fused, stream):
        if fused:
            fs.sample(x, self.W, temp, seed, step, out=(ids, mx), stream=stream)
        else:
            fs.sample_unfused(x, self.W, temp, seed, step, out=(ids, mx), stream=stream)

    def _body_graph(self, ids, stream):
        """The embedding of ``ids`` and the body, captured once as a CUDA graph
        (hundreds of small launches per step would otherwise be bound by the
        host's launch rate, not by the GPU).  Replaying it reads the current
        contents of ``ids`` and leaves the hidden state in the returned
        tensor."""
        torch = self.torch
        with torch.cuda.stream(stream):
            x = self.body(self.W[ids])                  # warm-up outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            x = self.body(self.W[ids])
        return graph, x

    def run(self, ids0, temp, steps, fused=True, seed=1234, warmup=3, stream=None):
        """``warmup`` + ``steps`` decode steps from token ids ``ids0`` [B]
        (int64, device): embed (rows of W), body, LM head + sampling; each
        step's sampled ids are the next step's input.

        The embedding and body are one CUDA-graph replay per step; the LM head
        is this library's call, with the step counter advancing.  Two timed
        passes on one stream: the whole loop between two events (nothing
        recorded between the launches) gives the step time; a second pass with
        events right before and after each step's LM-head call gives the head
        time.  Returns (StepTiming, the last step's ids)."""
        torch = self.torch
        stream = stream or torch.cuda.Stream()
        B = ids0.shape[0]
        ids = ids0.clone()
        mx = torch.empty(B, dtype=torch.float32, device=ids.device)
        graph, x = self._body_graph(ids, stream)
        ids.copy_(ids0)
        with torch.cuda.stream(stream):
            for i in range(warmup):
                graph.replay()
                self._head(x, temp, seed, i, ids, mx, fused, stream)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for i in range(steps):
                graph.replay()
                self._head(x, temp, seed, warmup + i, ids, mx, fused, stream)
            t1.record(stream)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
            for i, (a, b) in enumerate(ev):
                graph.replay()
                a.record(stream)
                self._head(x, temp, seed, warmup + steps + i, ids, mx, fused, stream)
                b.record(stream)
        torch.cuda.synchronize()
        del graph
        step_us = t0.elapsed_time(t1) / steps * 1e3
        head_us = sum(a.elapsed_time(b) for a, b in ev) / steps * 1e3
        return StepTiming(step_us, head_us), ids


def measure(W, batches=(1, 16, 256), layers=32, steps=10, warmup=3, layer=None, seed=1234):
    """Fused vs unfused LM-head sampling inside the decode loop, per batch.
    Returns one dict per batch size: step and head µs and the head's share of
    the step for both, and the step-time reduction fusion gives."""
    import torch
    loop = DecodeLoop(W, layers=layers, layer=layer)
    V = W.shape[0]
    out = []
    for B in batches:
        g = torch.Generator(device=W.device).manual_seed(B)
        ids0 = torch.randint(0, V, (B,), generator=g, device=W.device)
        temp = torch.ones(B, dtype=torch.float32, device=W.device)
        fused, _ = loop.run(ids0, temp, steps, fused=True, seed=seed, warmup=warmup)
        unf, _ = loop.run(ids0, temp, steps, fused=False, seed=seed, warmup=warmup)
        out.append({"B": B, "layers": layers,
                    "fused_step_us": round(fused.step_us, 1), "fused_head_us": round(fused.head_us, 1),
                    "fused_head_share": round(fused.share, 4),
                    "unfused_step_us": round(unf.step_us, 1), "unfused_head_us": round(unf.head_us, 1),
                    "unfused_head_share": round(unf.share, 4),
                    "step_time_reduction": round(1.0 - fused.step_us / unf.step_us, 4)})
    return out
