"""A small owner of the device buffers libdec needs, allocated through torch.

torch provides device memory and the stream; every step of the decoder runs
in libdec's kernels through the C ABI (``decoder_qwen3_step_gb300.dec``).
"""

from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import dec
from .inputs import BLOCK_TOKENS, LAYER_TENSORS, RMS_EPS, ROPE_BASE


def make_config(shape: dict, mode: int, max_positions: int) -> dec.dec_config:
    c = dec.dec_config()
    for k in ("vocab", "d_model", "n_layers", "n_heads", "n_kv_heads", "head_dim", "ff_hidden"):
        setattr(c, k, shape[k])
    c.max_positions = max_positions
    c.block_tokens = BLOCK_TOKENS
    c.mode = mode
    c.rope_base = ROPE_BASE
    c.rms_eps = RMS_EPS
    c.qk_norm = c.rope_split = c.tied = 1
    c.rope_scaling = c.sliding_window = c.attention_bias = 0
    return c


def _stream_ptr(stream) -> C.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


class Batch:
    """Host arrays of one step, kept alive while the C call reads them.

    Block tables may be Python lists or int32 numpy arrays; arrays are copied
    without a per-element conversion, which keeps a batch-32 decode step's
    marshalling near 40 us instead of about 200 us."""

    def __init__(self, seqs, device_ids: torch.Tensor | None = None):
        # seqs: list of (ids, start_position, block_table)
        self.n_seqs = len(seqs)
        if not seqs:  # an empty step: marshalled as is, the library refuses it
            seqs = [([], 0, [])]
        S = len(seqs)
        lens = [len(s[0]) for s in seqs]
        if all(n == 1 for n in lens):  # a decode step: one token per sequence
            self.seq_start = np.arange(S + 1, dtype=np.int32)
            self.ids = np.fromiter((s[0][0] for s in seqs), dtype=np.int32, count=S)
            self.positions = np.fromiter((s[1] for s in seqs), dtype=np.int32, count=S)
        else:
            self.seq_start = _i32(np.concatenate([[0], np.cumsum(lens)]))
            self.ids = _i32(np.concatenate([np.asarray(s[0]) for s in seqs]))
            self.positions = _i32(np.concatenate([s[1] + np.arange(n) for s, n in zip(seqs, lens)]))
        self.n_tokens = int(self.seq_start[-1])
        self.max_blocks = max(1, max(len(s[2]) for s in seqs))
        tab = np.zeros((S, self.max_blocks), dtype=np.int32)
        for i, s in enumerate(seqs):
            tab[i, : len(s[2])] = s[2]
        self.tables = tab
        self.device_ids = device_ids
        st = dec.dec_batch()
        st.n_seqs = self.n_seqs
        st.n_tokens = self.n_tokens
        st.ids = _ptr(self.ids) if device_ids is None else None
        st.ids_device = C.c_void_p(device_ids.data_ptr()) if device_ids is not None else None
        st.positions = _ptr(self.positions)
        st.seq_start = _ptr(self.seq_start)
        st.block_table = _ptr(self.tables)
        st.max_blocks = self.max_blocks
        self.struct = st


class Decoder:
    """A model + KV pool + workspace on one GPU, built from float32 weights."""

    def __init__(self, shape: dict, weights: dict, mode: int = dec.DEC_FP32, max_positions: int = 4096,
                 max_tokens: int = 4096, max_seqs: int = 64, n_blocks: int = 1024, device: str = "cuda:0",
                 stream=None):
        L = dec.lib()
        self.L = L
        self.shape = dict(shape)
        self.mode = mode
        self.device = torch.device(device)
        self.cfg = make_config(shape, mode, max_positions)
        self.max_tokens, self.max_seqs = max_tokens, max_seqs
        torch.cuda.set_device(self.device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        sz = C.c_size_t()
        dec.check(L.dec_weights_bytes(C.byref(self.cfg), C.byref(sz)), "dec_weights_bytes")
        self.packed = torch.empty(sz.value, dtype=torch.uint8, device=self.device)
        dec.check(L.dec_workspace_bytes(C.byref(self.cfg), max_tokens, max_seqs, C.byref(sz)), "dec_workspace_bytes")
        self.workspace = torch.empty(sz.value, dtype=torch.uint8, device=self.device)

        raw = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(self.device) for k, v in weights.items()}
        nl = shape["n_layers"]
        arrays = {}

        def per_layer(t):
            arr = (C.c_void_p * nl)(*[raw[f"layers.{l}.{t}"].data_ptr() for l in range(nl)])
            arrays[t] = arr
            return C.cast(arr, C.POINTER(C.c_void_p))

        w = dec.dec_weights()
        w.embed = raw["embed"].data_ptr()
        w.final_norm = raw["final_norm"].data_ptr()
        names = {"attn_norm": "attn_norm", "wq": "q", "wk": "k", "wv": "v", "q_norm": "q_norm", "k_norm": "k_norm",
                 "wo": "o", "mlp_norm": "mlp_norm", "w_gate": "gate", "w_up": "up", "w_down": "down"}
        assert set(names.values()) == set(LAYER_TENSORS)
        for field, t in names.items():
            setattr(w, field, per_layer(t))
        handle = C.c_void_p()
        dec.check(L.dec_create(C.byref(self.cfg), C.byref(w), C.c_void_p(self.packed.data_ptr()), self.packed.numel(),
                               C.c_void_p(self.workspace.data_ptr()), self.workspace.numel(), max_tokens, max_seqs,
                               _stream_ptr(self.stream), C.byref(handle)), "dec_create")
        self.handle = handle
        del raw, arrays

        dec.check(L.dec_pool_bytes(C.byref(self.cfg), n_blocks, C.byref(sz)), "dec_pool_bytes")
        self.slabs = torch.empty(sz.value, dtype=torch.uint8, device=self.device)
        pool = C.c_void_p()
        dec.check(L.dec_pool_create(C.byref(self.cfg), n_blocks, C.c_void_p(self.slabs.data_ptr()), self.slabs.numel(),
                                    C.byref(pool)), "dec_pool_create")
        self.pool = pool
        self.n_blocks = n_blocks

    # -- pool ---------------------------------------------------------------
    def alloc(self, n: int) -> list:
        ids = (C.c_int32 * max(n, 1))()
        dec.check(self.L.dec_pool_alloc(self.pool, n, ids), "dec_pool_alloc")
        return list(ids[:n])

    def release(self, ids) -> None:
        for i in ids:
            dec.check(self.L.dec_pool_release(self.pool, int(i)), "dec_pool_release")

    def free_blocks(self) -> int:
        n = C.c_int32()
        dec.check(self.L.dec_pool_free_blocks(self.pool, C.byref(n)), "dec_pool_free_blocks")
        return n.value

    def blocks_for(self, n_positions: int) -> list:
        return self.alloc((n_positions + BLOCK_TOKENS - 1) // BLOCK_TOKENS)

    # -- prefix cache ---------------------------------------------------------
    def prefix_keys(self, tokens) -> list:
        """Chained keys (dec_prefix_key) of the full blocks of a token sequence."""
        keys, prev = [], 0
        for i in range(len(tokens) // BLOCK_TOKENS):
            blk = (C.c_int32 * BLOCK_TOKENS)(*[int(t) for t in tokens[i * BLOCK_TOKENS:(i + 1) * BLOCK_TOKENS]])
            prev = self.L.dec_prefix_key(prev, blk, BLOCK_TOKENS)
            keys.append(prev)
        return keys

    def register_prefix(self, table, tokens) -> int:
        """Index the full blocks of a sequence whose K/V are written (positions
        0 .. len(tokens)-1 in `table`); returns how many blocks now carry their key."""
        n = 0
        for k, b in zip(self.prefix_keys(tokens), table):
            dec.check(self.L.dec_pool_set_fill(self.pool, int(b), BLOCK_TOKENS), "dec_pool_set_fill")
            ok = C.c_int32()
            dec.check(self.L.dec_pool_register(self.pool, int(b), k, C.byref(ok)), "dec_pool_register")
            n += ok.value
        return n

    def lookup_prefix(self, tokens) -> list:
        """Reacquire the cached blocks of the longest indexed prefix of tokens
        (whole blocks, stopping at the first miss); the caller releases them."""
        ids = []
        for k in self.prefix_keys(tokens):
            i = C.c_int32()
            dec.check(self.L.dec_pool_lookup(self.pool, k, C.byref(i)), "dec_pool_lookup")
            if i.value < 0:
                break
            ids.append(i.value)
        return ids

    def cached_blocks(self) -> int:
        n = C.c_int32()
        dec.check(self.L.dec_pool_cached_blocks(self.pool, C.byref(n)), "dec_pool_cached_blocks")
        return n.value

    # -- steps ----------------------------------------------------------------
    def prefill(self, seqs, rows: int = dec.DEC_ROWS_ALL, logits: bool = True, device_ids=None,
                out=None):
        """seqs: list of (ids, start, block_table).  Returns (logits [R,V] fp32 | None, argmax [R] int32)."""
        b = Batch(seqs, device_ids)
        R = b.n_tokens if rows == dec.DEC_ROWS_ALL else b.n_seqs
        lg, am = self._outputs(R, logits, out)
        dec.check(self.L.dec_prefill(self.handle, self.pool, C.byref(b.struct), rows,
                                     C.c_void_p(lg.data_ptr()) if lg is not None else None,
                                     C.c_void_p(am.data_ptr()), _stream_ptr(self.stream)), "dec_prefill")
        return lg, am

    def decode(self, seqs, logits: bool = True, device_ids=None, out=None):
        b = Batch(seqs, device_ids)
        lg, am = self._outputs(b.n_seqs, logits, out)
        dec.check(self.L.dec_decode(self.handle, self.pool, C.byref(b.struct),
                                    C.c_void_p(lg.data_ptr()) if lg is not None else None,
                                    C.c_void_p(am.data_ptr()), _stream_ptr(self.stream)), "dec_decode")
        return lg, am

    def _outputs(self, R, logits, out):
        if out is not None:
            return out
        V = self.shape["vocab"]
        lg = torch.empty((R, V), dtype=torch.float32, device=self.device) if logits else None
        am = torch.empty((R,), dtype=torch.int32, device=self.device)
        return lg, am

    def device_status(self) -> int:
        f = C.c_uint32()
        dec.check(self.L.dec_device_status(self.handle, C.byref(f)), "dec_device_status")
        return f.value

    def set_tensor_cores(self, on: bool) -> None:
        dec.check(self.L.dec_set_tensor_cores(self.handle, 1 if on else 0), "dec_set_tensor_cores")

    def set_graphs(self, on: bool) -> None:
        dec.check(self.L.dec_set_graphs(self.handle, 1 if on else 0), "dec_set_graphs")

    def set_megakernel(self, on: bool):
        """Serving-mode decode of <= 8 sequences as one persistent kernel (default on)."""
        dec.check(self.L.dec_set_megakernel(self.handle, 1 if on else 0), "dec_set_megakernel")

    def megakernel_available(self) -> bool:
        v = C.c_int32()
        dec.check(self.L.dec_megakernel_available(self.handle, C.byref(v)), "dec_megakernel_available")
        return bool(v.value)

    def set_dump(self, buf: torch.Tensor | None):
        if buf is None:
            dec.check(self.L.dec_set_dump(self.handle, None, 0), "dec_set_dump")
        else:
            dec.check(self.L.dec_set_dump(self.handle, C.c_void_p(buf.data_ptr()), buf.numel()), "dec_set_dump")

    def close(self):
        if getattr(self, "pool", None):
            self.L.dec_pool_destroy(self.pool)
            self.pool = None
        if getattr(self, "handle", None):
            self.L.dec_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def sampling_params(temperature=1.0, top_k=0, top_p=1.0, min_p=0.0, repetition_penalty=1.0, presence_penalty=0.0,
                    frequency_penalty=0.0) -> dec.dec_sampling:
    """One sequence's sampling parameters (the off values are the defaults)."""
    return dec.dec_sampling(float(temperature), int(top_k), float(top_p), float(min_p), float(repetition_penalty),
                            float(presence_penalty), float(frequency_penalty))


class DeviceHistory:
    """Prompt and output ids of a batch, already on the device (a serving loop
    appends each step's tokens there): ids [total] int32 on the device, host
    offsets [n + 1] and prompt counts [n]."""

    def __init__(self, histories, device="cuda"):
        flat, offs, npr = [], [0], []
        for pr, ou in histories:
            flat.extend(int(x) for x in pr)
            flat.extend(int(x) for x in ou)
            offs.append(len(flat))
            npr.append(len(pr))
        self.ids = torch.tensor(flat or [0], dtype=torch.int32, device=device)
        self.offsets = _i32(offs)
        self.n_prompt = _i32(npr or [0])


class Sampler:
    """The device sampler (libdec's dec_sample) with its workspace from torch.

    rng states live on the device as an int64 tensor [n, 2] (state, inc) whose
    bits are the C struct dec_rng; `streams(seeds)` makes the per-request
    streams of purpose 4.
    """

    def __init__(self, vocab: int, max_seqs: int, device="cuda"):
        self.L = dec.lib()
        self.device = torch.device(device)
        self.vocab, self.max_seqs = vocab, max_seqs
        nbytes = C.c_size_t()
        dec.check(self.L.dec_sampler_workspace_bytes(vocab, max_seqs, C.byref(nbytes)), "dec_sampler_workspace_bytes")
        self.ws = torch.empty(nbytes.value + 256, dtype=torch.uint8, device=self.device)
        base = self.ws.data_ptr()
        aligned = (base + 255) & ~255
        h = C.c_void_p()
        with torch.cuda.device(self.device):
            dec.check(self.L.dec_sampler_create(vocab, max_seqs, C.c_void_p(aligned), nbytes.value, C.byref(h)),
                      "dec_sampler_create")
        self.handle = h

    def streams(self, seeds, purpose: int = dec.DEC_PURPOSE_SAMPLE) -> torch.Tensor:
        out = np.zeros((len(seeds), 2), dtype=np.uint64)
        r = dec.dec_rng()
        for i, sd in enumerate(seeds):
            self.L.dec_rng_stream(C.c_uint64(int(sd) & (2**64 - 1)), C.c_uint64(purpose), C.byref(r))
            out[i] = (r.state, r.inc)
        return torch.from_numpy(out.view(np.int64)).to(self.device)

    def sample(self, logits: torch.Tensor, params, histories=None, rng: torch.Tensor | None = None, stream=None,
               out=None):
        """params: one dec_sampling per row of `logits` [n, >= vocab] (f32,
        on the device); histories: per row (prompt_ids, output_ids) or None.
        Returns device (tokens int32 [n], logprobs float64 [n]); `rng` is
        advanced in place."""
        n = logits.shape[0]
        assert logits.dtype == torch.float32 and logits.is_cuda and logits.stride(1) == 1
        P = (dec.dec_sampling * max(n, 1))(*params)
        offs = _i32([0] * (n + 1))
        npr = _i32([0] * max(n, 1))
        hist = None
        if isinstance(histories, DeviceHistory):
            hist, offs, npr = histories.ids, histories.offsets, histories.n_prompt
        elif histories is not None:
            flat = []
            for i, (pr, ou) in enumerate(histories):
                flat.extend(int(x) for x in pr)
                flat.extend(int(x) for x in ou)
                offs[i + 1] = len(flat)
                npr[i] = len(pr)
            if flat:
                hist = torch.tensor(flat, dtype=torch.int32, device=self.device)
        if out is None:
            tokens = torch.empty(n, dtype=torch.int32, device=self.device)
            logprobs = torch.empty(n, dtype=torch.float64, device=self.device)
        else:
            tokens, logprobs = out
        code = self.L.dec_sample(self.handle, C.c_void_p(logits.data_ptr()), logits.stride(0), n, P,
                                 C.c_void_p(hist.data_ptr() if hist is not None else 0), _ptr(offs), _ptr(npr),
                                 C.c_void_p(rng.data_ptr()), C.c_void_p(tokens.data_ptr()),
                                 C.c_void_p(logprobs.data_ptr()), _stream_ptr(stream))
        dec.check(code, "dec_sample")
        if hist is not None and stream is not None:
            hist.record_stream(stream)  # the allocator must not reuse it before `stream` has read it
        self._keep = hist
        return tokens, logprobs

    def status(self) -> int:
        f = C.c_uint32()
        dec.check(self.L.dec_sampler_status(self.handle, C.byref(f)), "dec_sampler_status")
        return f.value

    def close(self):
        if getattr(self, "handle", None):
            self.L.dec_sampler_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
