"""TACO's compressed two-shot AllReduce among R logical ranks on one GPU.

The two-shot AllReduce of the TACO pages (gist.science pt summary, §2.B.3:
ReduceScatter + AllGather with the compression operator between the phases)
over R ranks whose tensors all live on this GPU. Nothing here computes:
every step is a libtaco call, and the two exchanges are pointer
permutations, which is what the receive buffers of a real ReduceScatter and
AllGather would hand to the same calls.

  rank r:  X_r [M, h] = R row chunks of [M/R, h]
  1. compress      rank r compresses its R chunks         (taco_compress_shards_mma,
                                                           or taco_compress_shards_fwht)
  2. ReduceScatter rank c receives chunk c of every rank  (pointers)
  3. reduce        rank c sums and recompresses them      (taco_reduce_recompress_ptrs)
  4. AllGather     every rank receives the R results      (pointers)
  5. expand        the R chunks to the full [M, h] result (taco_decompress_shards_ptrs)

All ranks end with the same tensor, so step 5 runs once. When R * R <= 16
(the shard limit of one launch) step 1 is a single compress launch over the
R * R chunks of all ranks and steps 2-3 a single batched reduce-recompress
launch (one grid row per destination rank): 3 launches in all, else 2 R + 1.
"""

from __future__ import annotations

import torch

from . import binding as tb


class EmulatedTwoShotAllReduce:
    """Preallocated buffers and the launch sequence of one compressed AllReduce."""

    def __init__(self, R: int, M: int, h: int, block: int,
                 target_energy: float = tb.DEFAULT_TARGET_ENERGY, variant: int = tb.VARIANT_DUAL,
                 device="cuda", compress: str = "mma", fmt: str = "e4m3"):
        """compress: "mma" (tensor-core Hadamard) or "fwht" (CUDA-core FWHT);
        fmt: "e4m3" (FP8 codes) or "int8" (the INT8 fallback format; its
        compress runs on the tensor cores)."""
        if not 1 <= R <= tb.MAX_SHARDS:
            raise ValueError(f"R must be in 1..{tb.MAX_SHARDS}")
        if compress not in ("mma", "fwht"):
            raise ValueError('compress must be "mma" or "fwht"')
        if fmt not in ("e4m3", "int8"):
            raise ValueError('fmt must be "e4m3" or "int8"')
        self.fmt = fmt
        if fmt == "int8":
            self._compress = tb.taco_compress_shards_int8
            self._recompress = tb.taco_reduce_recompress_int8_ptrs
            self._expand = tb.taco_decompress_shards_int8_ptrs
            self._format = tb.FORMAT_INT8
        else:
            self._compress = tb.taco_compress_shards_mma if compress == "mma" else tb.taco_compress_shards_fwht
            self._recompress = tb.taco_reduce_recompress_ptrs
            self._expand = tb.taco_decompress_shards_ptrs
            self._format = tb.FORMAT_E4M3
        if M % R:
            raise ValueError("M must be a multiple of R")
        self.R, self.M, self.h, self.block = R, M, h, block
        self.chunk = M // R
        self.target_energy, self.variant = float(target_energy), variant
        dev = torch.device(device)
        sb = tb.shard_bytes(self.chunk, h, block)
        self.batched = R * R <= tb.MAX_SHARDS
        # rank r's compressed chunks are rows r*R .. r*R+R-1 of one bundle
        self.bundle_all = torch.empty((R * R, sb), dtype=torch.uint8, device=dev)
        self.headers_all = torch.empty((R * R, tb.HEADER_BYTES), dtype=torch.uint8, device=dev)
        self.bundles = [self.bundle_all[r * R:(r + 1) * R] for r in range(R)]
        self.headers = [self.headers_all[r * R:(r + 1) * R] for r in range(R)]
        self.reduced_all = torch.empty((R, sb), dtype=torch.uint8, device=dev)
        self.reduced_headers_all = torch.empty((R, tb.HEADER_BYTES), dtype=torch.uint8, device=dev)
        self.reduced = [self.reduced_all[d] for d in range(R)]
        self.reduced_headers = [self.reduced_headers_all[d] for d in range(R)]
        self.out = torch.empty((M, h), dtype=torch.bfloat16, device=dev)
        self.workspace = tb.new_workspace(R * R if self.batched else R, dev)
        self._graph = None

    def launches(self) -> int:
        """Kernel launches of one AllReduce."""
        return 3 if self.batched else 2 * self.R + 1

    def __call__(self, xs: torch.Tensor, stream=None) -> torch.Tensor:
        """xs: bf16 [R, M, h], rank r's tensor in xs[r]. Returns the reduced [M, h]."""
        R, c, h, n = self.R, self.chunk, self.h, self.block
        if xs.shape != (R, self.M, h) or xs.dtype != torch.bfloat16 or not xs.is_contiguous():
            raise ValueError(f"xs must be a contiguous bf16 tensor of shape {(R, self.M, h)}")
        if self.batched:                                              # 1. compress
            self._compress(xs.view(R * R, c, h), n, self.target_energy, self.variant,
                           bundle=self.bundle_all, headers=self.headers_all,
                           workspace=self.workspace, stream=stream)
        else:
            for r in range(R):
                self._compress(xs[r].view(R, c, h), n, self.target_energy, self.variant,
                               bundle=self.bundles[r], headers=self.headers[r],
                               workspace=self.workspace, stream=stream)
        if self.batched:                                              # 2.+3. reduce-scatter
            received = [self.bundles[r][dst] for dst in range(R) for r in range(R)]
            tb.taco_reduce_recompress_batched_ptrs(received, R, c, h, n, self.target_energy, self.variant,
                                                   self._format, shards_out=self.reduced_all,
                                                   headers=self.reduced_headers_all,
                                                   workspace=self.workspace, stream=stream)
        else:
            for dst in range(R):
                received = [self.bundles[r][dst] for r in range(R)]
                self._recompress(received, c, h, n, self.target_energy, self.variant,
                                 shard=self.reduced[dst], header=self.reduced_headers[dst],
                                 workspace=self.workspace, stream=stream)
        self._expand(self.reduced, c, h, n,                           # 4.+5. all-gather
                     out=self.out.view(R, c, h), stream=stream)
        return self.out

    def capture(self, xs: torch.Tensor) -> torch.cuda.CUDAGraph:
        """Record one AllReduce of `xs` (fixed address) into a CUDA graph.

        Call the object once outside capture first: the library's one-time
        per-device set-up cannot run inside a capture.
        """
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self(xs)
        self._graph = g
        return g


class PipelinedTwoShotAllReduce:
    """The same compressed two-shot AllReduce cut into S row segments that flow
    through compress, reduce-recompress and expand on three streams.

    TACO overlaps the compression with the ReduceScatter and AllGather phases
    (gist.science pt summary, §2.B.3). Here the phases are launches on one
    GPU: segment j is compressed on the caller's stream while segment j - 1
    is reduced and recompressed on a second stream and segment j - 2 is
    expanded on a third; events order each segment's three steps. Every
    block's arithmetic is the serial AllReduce's (blocks never straddle rows
    and the R shards of a block are summed in the same order), so the result
    is bit for bit the serial one. The three streams fork from and join the
    caller's stream, so one call can be captured in a CUDA graph.

    Per segment: R compress launches (rank r's R chunks of the segment are
    one contiguous [R, M/(S R), h] tensor), ceil(R / Y) batched
    reduce-recompress launches (Y destination ranks each, Y R <= 16 shards)
    and one expand launch.
    """

    def __init__(self, R: int, M: int, h: int, block: int, segments: int = 4,
                 target_energy: float = tb.DEFAULT_TARGET_ENERGY, variant: int = tb.VARIANT_DUAL,
                 device="cuda", fmt: str = "e4m3"):
        if not 1 <= R <= tb.MAX_SHARDS:
            raise ValueError(f"R must be in 1..{tb.MAX_SHARDS}")
        if segments < 1 or M % (R * segments):
            raise ValueError("M must be a multiple of R * segments")
        if fmt not in ("e4m3", "int8"):
            raise ValueError('fmt must be "e4m3" or "int8"')
        self._compress = tb.taco_compress_shards_int8 if fmt == "int8" else tb.taco_compress_shards_mma
        self._expand = tb.taco_decompress_shards_int8_ptrs if fmt == "int8" else tb.taco_decompress_shards_ptrs
        self._format = tb.FORMAT_INT8 if fmt == "int8" else tb.FORMAT_E4M3
        self.R, self.M, self.h, self.block, self.S = R, M, h, block, segments
        self.seg_rows = M // segments
        self.chunk = self.seg_rows // R
        self.target_energy, self.variant = float(target_energy), variant
        dev = torch.device(device)
        sb = tb.shard_bytes(self.chunk, h, block)
        S = segments
        self.bundles = torch.empty((S, R, R, sb), dtype=torch.uint8, device=dev)    # [segment][rank][chunk]
        self.headers = torch.empty((S, R, R, tb.HEADER_BYTES), dtype=torch.uint8, device=dev)
        self.Y = max(1, min(R, tb.MAX_SHARDS // R))                                  # reductions per launch
        self.reduced = torch.empty((S, R, sb), dtype=torch.uint8, device=dev)
        self.reduced_headers = torch.empty((S, R, tb.HEADER_BYTES), dtype=torch.uint8, device=dev)
        self.out = torch.empty((M, h), dtype=torch.bfloat16, device=dev)
        self.ws_compress = tb.new_workspace(R, dev)         # launches in order on one stream
        self.ws_reduce = tb.new_workspace(self.Y, dev)
        self.s_reduce = torch.cuda.Stream(dev)
        self.s_expand = torch.cuda.Stream(dev)
        self.ev_compressed = [torch.cuda.Event() for _ in range(S)]
        self.ev_reduced = [torch.cuda.Event() for _ in range(S)]

    def launches(self) -> int:
        """Kernel launches of one AllReduce."""
        return self.S * (self.R + -(-self.R // self.Y) + 1)

    def __call__(self, xs: torch.Tensor, stream=None) -> torch.Tensor:
        """xs: bf16 [R, M, h], rank r's tensor in xs[r]. Returns the reduced [M, h]."""
        R, c, h, n, rows = self.R, self.chunk, self.h, self.block, self.seg_rows
        if xs.shape != (R, self.M, h) or xs.dtype != torch.bfloat16 or not xs.is_contiguous():
            raise ValueError(f"xs must be a contiguous bf16 tensor of shape {(R, self.M, h)}")
        s_c = stream or torch.cuda.current_stream()
        self.s_reduce.wait_stream(s_c)                       # fork: the inputs are ready
        self.s_expand.wait_stream(s_c)
        for j in range(self.S):
            for r in range(R):                               # 1. compress (caller's stream)
                self._compress(xs[r, j * rows:(j + 1) * rows].view(R, c, h), n, self.target_energy,
                               self.variant, bundle=self.bundles[j, r], headers=self.headers[j, r],
                               workspace=self.ws_compress, stream=s_c)
            self.ev_compressed[j].record(s_c)
            self.s_reduce.wait_event(self.ev_compressed[j])  # 2.+3. reduce-scatter (second stream)
            for d0 in range(0, R, self.Y):
                dests = range(d0, min(R, d0 + self.Y))
                received = [self.bundles[j, r, d] for d in dests for r in range(R)]
                tb.taco_reduce_recompress_batched_ptrs(
                    received, len(dests), c, h, n, self.target_energy, self.variant, self._format,
                    shards_out=self.reduced[j, d0:d0 + len(dests)],
                    headers=self.reduced_headers[j, d0:d0 + len(dests)],
                    workspace=self.ws_reduce, stream=self.s_reduce)
            self.ev_reduced[j].record(self.s_reduce)
            self.s_expand.wait_event(self.ev_reduced[j])     # 4.+5. all-gather (third stream)
            self._expand([self.reduced[j, d] for d in range(R)], c, h, n,
                         out=self.out[j * rows:(j + 1) * rows].view(R, c, h), stream=self.s_expand)
        s_c.wait_stream(self.s_reduce)                       # join
        s_c.wait_stream(self.s_expand)
        return self.out

    def capture(self, xs: torch.Tensor) -> torch.cuda.CUDAGraph:
        """Record one AllReduce of `xs` (fixed address) into a CUDA graph
        (call the object once outside capture first)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self(xs)
        return g
