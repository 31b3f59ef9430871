"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and put its
results next to the oracle's, on identical seeded inputs."""
import numpy as np

import oracle
from quantized_q8_activation_quantize_gb300 import binding as B

# the parity bar: max |Y_gpu - Y_ref| / ||Y_ref[m, :]||_2  (row-L2-normalised relative error)
REL_TOL = 1e-3


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_plane(x, rms_w=None, eps=1e-6, plane=None):
    """Quantize x [M, K] (f32) on the GPU; returns (plane tensor, logical (q16, q8, d, S) as numpy)."""
    import torch
    M, K = x.shape
    xd = dev(x.astype(np.float32))
    wd = dev(rms_w.astype(np.float32)) if rms_w is not None else None
    if plane is None:
        plane = B.alloc_plane(M, K)
    B.mq_quantize_q8(xd, M, K, wd, eps, plane)
    torch.cuda.synchronize()
    B.mq_device_status()
    q16, q8, d, s = B.plane_views(plane, M, K)
    return plane, (q16.float().cpu().numpy(), q8.cpu().numpy(), d.t().contiguous().cpu().numpy(),
                   s.t().contiguous().cpu().numpy())


def assert_plane_equal(got, ref):
    q16, q8, d, s = got
    q, dr, sr = ref
    assert np.array_equal(q8, q), f"int8 codes differ at {np.argwhere(q8 != q)[:5]}"
    assert np.array_equal(q16, q.astype(np.float32)), "f16 codes differ from the int8 codes"
    assert np.array_equal(d.view(np.uint32), dr.view(np.uint32)), f"scales differ at {np.argwhere(d != dr)[:5]}"
    assert np.array_equal(s, sr), "block sums differ"


def _tf32_rna(a):
    """f32 -> the nearest tf32 value (10 explicit mantissa bits), ties away from zero, kept as f32."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((b + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def assert_ds_consistent(plane, M, K):
    """The plane's ds section holds, per block, the tf32 pair of the f32 product d * S (the
    definition in include/mq.h): hi = tf32(d * S), lo = tf32(d * S - hi), laid out per super-block
    of a token as hi[8] then lo[8]."""
    _, _, d, s, ds = B.plane_views(plane, M, K, with_ds=True)
    d = d.t().contiguous().cpu().numpy()
    s = s.t().contiguous().cpu().numpy()
    ds = ds.cpu().numpy().reshape(M, K // 256, 2, 8)
    p = (d * s.astype(np.float32)).astype(np.float32)
    hi = _tf32_rna(p)
    lo = _tf32_rna((p - hi).astype(np.float32))
    assert np.array_equal(ds[:, :, 0, :].reshape(M, -1).view(np.uint32), hi.view(np.uint32)), "ds hi differs"
    assert np.array_equal(ds[:, :, 1, :].reshape(M, -1).view(np.uint32), lo.view(np.uint32)), "ds lo differs"


def run_matmul(path, fmt, w, plane, M, K, N):
    import torch
    wd = dev(w.reshape(N, -1))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    {"gemm": B.GEMM, "gemv": B.GEMV, "small": B.GEMM_SMALL}[path][fmt](wd, N, K, plane, M, y)
    torch.cuda.synchronize()
    B.mq_device_status()
    return y.cpu().numpy(), wd


def run_dump(path, fmt, wd, plane, M, K, N, m0, mc, n0, nc):
    import torch
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    I = torch.full((mc, nc, K // 32), -7, dtype=torch.int32, device="cuda")
    op = B.DEBUG_OP[(path, fmt)]
    B.mq_debug_blockdots(op, wd, N, K, plane, M, y, m0, mc, n0, nc, I)
    torch.cuda.synchronize()
    B.mq_device_status()
    return I.cpu().numpy(), y.cpu().numpy()


def rel_err(y, ref, rows=None):
    """max over the compared entries of |y - ref| / ||ref_full[m, :]||_2 (row norms from `rows` if given)."""
    norms = np.linalg.norm(ref if rows is None else rows, axis=1, keepdims=True)
    norms = np.where(norms == 0, 1.0, norms)
    return float((np.abs(y.astype(np.float64) - ref) / norms).max())


def oracle_plane(x, rms_w=None, eps=1e-6):
    return oracle.quantize_q8(x, rms_w, eps)
