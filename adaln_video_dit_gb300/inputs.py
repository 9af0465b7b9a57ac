"""Seeded synthetic inputs for the fused AdaLN operator.

This module draws random inputs and packs them; it holds none of the
operator's arithmetic.  Both the CUDA path and the CPU oracle are fed from it,
with identical bits: floating-point tensors are drawn in float32, and for bf16
workloads rounded to bf16 (round to nearest, ties to even) here, once, and
handed to both sides as raw uint16 bits.

Workloads (shapes and value distributions of AdaptiveLoad's experiments:
"Technical summary" section 4, Wan 2.1 on a mixed image/video corpus; the
corpus itself is not available, so these synthetic draws stand in for it):

  1 tiny_fp32    T=256, D=128, fp32, 1 segment.  x ~ N(0,1) + per-row U(-3,3)
                 offset; shift, scale ~ N(0, 0.1); dy ~ N(0, 1).
  2 wan13b       T=8192 (2 x 4096), D=1536, bf16, 2 segments.  x ~ N(0,1) times
                 a per-row factor U(0.5, 4); shift, scale ~ N(0, 0.5);
                 dy ~ N(0, 1e-2).
  3 long_video   T=32760 (21 x 30 x 52), D=5120, bf16, 1 segment.  x ~ N(0,1)
                 with round(0.001 D) outlier channels (seeded, fixed across rows)
                 scaled by 50; shift, scale ~ N(0, 0.5); dy ~ N(0, 1e-2).
  4 mixed_varlen D=3072, bf16.  8 bucket draws of a length S from
                 {256, 1024, 4096, 16384, 32760} with probabilities
                 {.4, .25, .2, .1, .05}; each draw adds B_shape(S) samples of
                 length S, B_shape = max(1, min(M_mem // S, M_comp // S**2)) with
                 M_mem = 65536 and M_comp = 2**31 (section 2.A, dual-constraint
                 bucketing, p = 2).  Samples are packed contiguously in draw
                 order; seg_id = running sample index.  x ~ N(0,1);
                 shift, scale [nseg, D] ~ N(0, 0.5); dy ~ N(0, 1e-2).
  5 mmdit_joint  8 samples, each 512 text + 4096 video tokens (T=36864),
                 D=3072, bf16; seg_id = 2*sample + (0 text, 1 video), 16
                 segments; 60 modulation sites (2 per block x 30 blocks), each
                 with its own shift, scale ~ N(0, 0.5); x ~ N(0,1);
                 dy ~ N(0, 1e-2).

The second parameter of N(., .) is the standard deviation.  eps = 1e-6.
"""
import numpy as np

EPS = 1e-6

NAMES = {1: "tiny_fp32", 2: "wan13b", 3: "long_video", 4: "mixed_varlen",
         5: "mmdit_joint"}

# Rows drawn per chunk when generating large tensors (bounds temporaries).
_CHUNK_ELEMS = 1 << 24


def to_bf16_bits(a):
    """Round float32 to bf16 (nearest, ties to even); return uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b):
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rngs(seed, n):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def _normal_rows(rng, T, D, std, out_bf16, row_factor=None, col_factor=None):
    """[T, D] of N(0, std), drawn row-chunk by row-chunk in float32."""
    out = np.empty((T, D), np.uint16 if out_bf16 else np.float32)
    step = max(1, _CHUNK_ELEMS // max(D, 1))
    for r0 in range(0, T, step):
        r1 = min(T, r0 + step)
        a = rng.standard_normal((r1 - r0, D), dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        if row_factor is not None:
            a *= row_factor[r0:r1, None]
        if col_factor is not None:
            a *= col_factor[None, :]
        out[r0:r1] = to_bf16_bits(a) if out_bf16 else a
    return out


def b_shape(S, m_mem=65536, m_comp=2 ** 31, p=2):
    """Bucket batch size of the dual-constraint scheduler (section 2.A)."""
    return max(1, min(m_mem // S, m_comp // S ** p))


def mixed_varlen_lengths(seed=4, draws=8):
    """Per-sample lengths of workload 4, in packing order."""
    rng = np.random.default_rng(np.random.SeedSequence(seed).spawn(1)[0])
    buckets = np.array([256, 1024, 4096, 16384, 32760])
    probs = np.array([0.4, 0.25, 0.2, 0.1, 0.05])
    lengths = []
    for S in rng.choice(buckets, size=draws, p=probs):
        lengths += [int(S)] * b_shape(int(S))
    return lengths


def seg_ids_from_lengths(lengths):
    return np.repeat(np.arange(len(lengths), dtype=np.int32),
                     np.asarray(lengths, dtype=np.int64))


def make(config, *, sites=1, T_override=None):
    """Draw the inputs of workload `config` (1..5).

    Returns a dict: name, dtype ('f32' or 'bf16'), T, D, nseg, eps,
    x, dy [T, D]; shift, scale [nseg, D] (for workload 5 with sites > 1,
    lists of `sites` arrays); seg_id int32 [T].  bf16 tensors are uint16 bits.
    T_override truncates workloads 2-3 to their first rows (small tests).
    """
    name = NAMES[config]
    if config == 1:
        rx, rm, rd, ro = _rngs(1, 4)
        T, D, nseg, bf = 256, 128, 1, False
        x = rx.standard_normal((T, D), dtype=np.float32)
        x += ro.uniform(-3.0, 3.0, size=(T, 1)).astype(np.float32)
        shift = (rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.1))
        scale = (rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.1))
        dy = rd.standard_normal((T, D), dtype=np.float32)
        seg_id = np.zeros(T, np.int32)
    elif config == 2:
        rx, rm, rd, ro = _rngs(2, 4)
        T, D, nseg, bf = 8192, 1536, 2, True
        r = ro.uniform(0.5, 4.0, size=T).astype(np.float32)
        seg_id = seg_ids_from_lengths([4096, 4096])
        if T_override:
            T = T_override
            r, seg_id = r[:T], seg_id[:T]
        x = _normal_rows(rx, T, D, 1.0, bf, row_factor=r)
        shift = to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5))
        scale = to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5))
        dy = _normal_rows(rd, T, D, 1e-2, bf)
    elif config == 3:
        rx, rm, rd, ro = _rngs(3, 4)
        T, D, nseg, bf = 32760, 5120, 1, True
        if T_override:
            T = T_override
        n_out = int(round(0.001 * D))
        col = np.ones(D, np.float32)
        col[ro.choice(D, size=n_out, replace=False)] = 50.0
        x = _normal_rows(rx, T, D, 1.0, bf, col_factor=col)
        shift = to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5))
        scale = to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5))
        dy = _normal_rows(rd, T, D, 1e-2, bf)
        seg_id = np.zeros(T, np.int32)
    elif config == 4:
        rx, rm, rd = _rngs(40, 3)
        D, bf = 3072, True
        seg_id = seg_ids_from_lengths(mixed_varlen_lengths(4))
        T, nseg = int(seg_id.shape[0]), int(seg_id[-1]) + 1
        x = _normal_rows(rx, T, D, 1.0, bf)
        shift = to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5))
        scale = to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5))
        dy = _normal_rows(rd, T, D, 1e-2, bf)
    elif config == 5:
        rx, rm, rd = _rngs(5, 3)
        D, bf, nseg = 3072, True, 16
        lengths = [512, 4096] * 8
        seg_id = seg_ids_from_lengths(lengths)
        T = int(seg_id.shape[0])
        x = _normal_rows(rx, T, D, 1.0, bf)
        shift, scale = [], []
        for _ in range(sites):
            shift.append(to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5)))
            scale.append(to_bf16_bits(rm.standard_normal((nseg, D), dtype=np.float32) * np.float32(0.5)))
        if sites == 1:
            shift, scale = shift[0], scale[0]
        dy = _normal_rows(rd, T, D, 1e-2, bf)
    else:
        raise ValueError(f"unknown workload {config}")
    return dict(name=name, config=config, dtype="bf16" if bf else "f32",
                T=int(T), D=int(D), nseg=int(nseg), eps=EPS, x=x, dy=dy,
                shift=shift, scale=scale, seg_id=seg_id)


def random_case(seed, T, D, nseg, dtype="bf16", lengths=None, x_std=1.0,
                mod_std=0.5, dy_std=1e-2):
    """Small generic case for edge tests: contiguous segments of the given
    lengths (random split of T into nseg parts, some possibly empty, when
    lengths is None)."""
    rx, rm, rd, rl = _rngs(seed, 4)
    if lengths is None:
        cuts = np.sort(rl.integers(0, T + 1, size=nseg - 1))
        lengths = np.diff(np.concatenate([[0], cuts, [T]])).tolist()
    assert sum(lengths) == T and len(lengths) == nseg
    seg_id = seg_ids_from_lengths(lengths)
    bf = dtype == "bf16"
    x = _normal_rows(rx, T, D, x_std, bf)
    dy = _normal_rows(rd, T, D, dy_std, bf)
    shift = _normal_rows(rm, nseg, D, mod_std, bf)
    scale = _normal_rows(rm, nseg, D, mod_std, bf)
    return dict(name=f"random_{seed}", config=0, dtype=dtype, T=T, D=D,
                nseg=nseg, eps=EPS, x=x, dy=dy, shift=shift, scale=scale,
                seg_id=seg_id)
