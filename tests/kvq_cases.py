"""Case builders shared by the GPU parity tests: seeded inputs, the oracle's
cache bytes and expected outputs, and the same inputs on the device."""
import numpy as np
import torch

import oracle
from quantized_paged_kv_reshape_gb300 import ops
from quantized_paged_kv_reshape_gb300 import workloads as W

ALL_FORMATS = list(oracle.FORMATS)
DEC_TOL_MAX, DEC_TOL_MEAN = 2e-3, 2e-4


def bf16_round(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def fp8_scales(k, v):
    return float(np.abs(k).max()) / 448.0, float(np.abs(v).max()) / 448.0


def decode_case(fmt, lens, nq, nkv, hd, bs=16, seed=0, in_dtype="f32", spare=3,
                outliers=True, stride_pad=0):
    """Seeded paged cache written by the oracle; returns a dict of host arrays."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in lens]
    nb_need = sum(-(-n // bs) for n in lens)
    num_blocks = nb_need + spare
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(1, max(-(-n // bs) for n in lens))
    tables = np.full((len(lens), mb), -1, np.int32)
    cur = 0
    for s, n in enumerate(lens):
        nb = -(-n // bs)
        tables[s, :nb] = perm[cur:cur + nb]
        cur += nb
    total = sum(lens)
    ch = np.ones((nkv, hd), np.float32)
    if outliers:
        for h in range(nkv):
            ch[h, rng.choice(hd, 2, replace=False)] = 8.0
    k = rng.standard_normal((total, nkv, hd)).astype(np.float32) * ch
    v = rng.standard_normal((total, nkv, hd)).astype(np.float32) * ch
    q = rng.standard_normal((len(lens), nq, hd)).astype(np.float32)
    if in_dtype == "bf16":
        k, v, q = bf16_round(k), bf16_round(v), bf16_round(q)
    slots = np.concatenate([tables[s, np.arange(n) // bs].astype(np.int64) * bs + np.arange(n) % bs
                            for s, n in enumerate(lens) if n > 0] or [np.zeros(0, np.int64)])
    kside, vside = oracle.kv_pair(fmt)
    ks, vs = fp8_scales(k, v) if total else (1.0, 1.0)
    kst = (oracle.block_bytes(kside, bs, nkv, hd) + 15) // 16 * 16 + stride_pad
    vst = (oracle.block_bytes(vside, bs, nkv, hd) + 15) // 16 * 16 + stride_pad
    kc = np.zeros(num_blocks * kst, np.uint8)
    vc = np.zeros(num_blocks * vst, np.uint8)
    if total:
        oracle.cache_write(kside, k, kc, slots, nkv, hd, bs, kst, scale=ks)
        oracle.cache_write(vside, v, vc, slots, nkv, hd, bs, vst, scale=vs)
    return dict(fmt=fmt, lens=np.array(lens, np.int32), nq=nq, nkv=nkv, hd=hd, bs=bs,
                tables=tables, k=k, v=v, q=q, slots=slots, kc=kc, vc=vc, kst=kst, vst=vst,
                k_scale=ks, v_scale=vs, num_blocks=num_blocks, in_dtype=in_dtype)


def oracle_decode(c, window=0, sparse=0.0, q=None):
    return oracle.paged_decode(c["q"] if q is None else q, c["kc"], c["vc"], c["tables"],
                               c["lens"], c["nkv"], c["hd"], c["bs"], c["kst"], c["vst"],
                               c["fmt"], k_scale=c["k_scale"], v_scale=c["v_scale"],
                               window=window, sparse_v_threshold=sparse)


def gpu_decode(c, window=0, sparse=0.0, dev="cuda", out_dtype=torch.float32, q_dtype=None,
               err=None, workspace=None):
    kpool = torch.from_numpy(c["kc"].reshape(c["num_blocks"], c["kst"])).to(dev)
    vpool = torch.from_numpy(c["vc"].reshape(c["num_blocks"], c["vst"])).to(dev)
    qd = q_dtype or (torch.bfloat16 if c["in_dtype"] == "bf16" else torch.float32)
    q = torch.from_numpy(c["q"]).to(dev).to(qd)
    out = ops.paged_decode(q, kpool, vpool, torch.from_numpy(c["tables"]).to(dev),
                           torch.from_numpy(c["lens"]).to(dev), c["fmt"], c["nkv"], c["bs"],
                           out_dtype=out_dtype, k_scale=c["k_scale"], v_scale=c["v_scale"],
                           sliding_window=window, sparse_v_threshold=sparse, error_flag=err,
                           workspace=workspace)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def assert_decode_close(got, ref, tol_max=DEC_TOL_MAX, tol_mean=DEC_TOL_MEAN):
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert err.max() <= tol_max, f"max-abs {err.max():.3e}"
    assert err.mean() <= tol_mean, f"mean-abs {err.mean():.3e}"
    return err.max(), err.mean()
