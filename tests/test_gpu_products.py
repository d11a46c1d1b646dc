"""Each weight-product kernel alone, through the C ABI test hook
dec_debug_product: Y = X W^T for every packed matrix of a layer and the
embedding, on the CUDA-core kernels (few and many token rows) and on the
tcgen05 kernel, against float64 numpy on the very same bf16 / fp32 values.
A transposed operand, a skipped K block, a wrong swizzle or a wrong
gate/up interleave is an O(1) error here; the bound only admits fp32
summation-order noise."""

import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402
from decoder_qwen3_step_gb300.runtime import Decoder  # noqa: E402
from oracle.numerics import bf16_round  # noqa: E402

pytestmark = pytest.mark.gpu


def packed_matrix(w, shape, which, layer):
    """The matrix as the library packs it (rows in packed order), float64."""
    p = f"layers.{layer}."
    if which == 0:
        return np.concatenate([w[p + "q"], w[p + "k"], w[p + "v"]])
    if which == 1:
        return w[p + "o"]
    if which == 2:
        g, u = w[p + "gate"], w[p + "up"]
        F = g.shape[0]
        out = np.empty((2 * F, g.shape[1]), dtype=g.dtype)
        for grp in range(F // 8):
            out[16 * grp:16 * grp + 8] = g[8 * grp:8 * grp + 8]
            out[16 * grp + 8:16 * grp + 16] = u[8 * grp:8 * grp + 8]
        return out
    if which == 3:
        return w[p + "down"]
    return w["embed"]


def run_product(m, which, layer, X, path):
    T = X.shape[0]
    rows = {0: (m.shape["n_heads"] + 2 * m.shape["n_kv_heads"]) * m.shape["head_dim"], 1: m.shape["d_model"],
            2: 2 * m.shape["ff_hidden"], 3: m.shape["d_model"], 4: m.shape["vocab"]}[which]
    Y = torch.full((T, rows), float("nan"), dtype=torch.float32, device=m.device)
    s = torch.cuda.current_stream()
    dec.check(m.L.dec_debug_product(m.handle, which, layer, C.c_void_p(X.data_ptr()), T, C.c_void_p(Y.data_ptr()),
                                    path, C.c_void_p(s.cuda_stream)), "dec_debug_product")
    torch.cuda.synchronize()
    return Y.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_every_product_against_float64(mode):
    shape = inputs.SHAPES["small"]
    w = inputs.make_weights(shape)
    m = Decoder(shape, w, mode=dec.DEC_BF16_F16KV if mode == "bf16" else dec.DEC_FP32, max_positions=256,
                max_tokens=512, max_seqs=4, n_blocks=16)
    rng = np.random.default_rng(11)
    layer = 5
    for which in range(5):
        W = packed_matrix(w, shape, which, layer)
        if mode == "bf16":
            W = bf16_round(W)
        W = W.astype(np.float64)
        K = W.shape[1]
        for T in (1, 7, 32, 300):
            Xf = rng.standard_normal((T, K)).astype(np.float32)
            if mode == "bf16":
                Xf = bf16_round(Xf)
                X = torch.from_numpy(Xf).to(torch.bfloat16).cuda()
            else:
                X = torch.from_numpy(Xf).cuda()
            ref = Xf.astype(np.float64) @ W.T
            scale = np.abs(Xf).astype(np.float64) @ np.abs(W).T  # bound on the rounding of each sum
            paths = [0]
            if mode == "bf16" and W.shape[0] % 128 == 0:
                paths.append(1 if T > 32 else 2)
            for path in paths:
                Y = run_product(m, which, layer, X, path)
                err = np.abs(Y - ref) / np.maximum(scale, 1e-30)
                assert np.isfinite(Y).all(), (which, T, path)
                assert err.max() < 2e-6, (which, T, path, float(err.max()))
    assert m.device_status() == 0
    m.close()
