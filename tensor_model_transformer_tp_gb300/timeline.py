"""Per-CTA timelines of the library's tensor-core kernels (a debugging aid).

Reads the globaltimer stamps that the kernels write when a timeline buffer is
installed (``oases_debug_gemm_timeline``, ``oases_debug_attention_timeline``)
and prints where a launch spends its time.  Needs a GPU and the built library.

    python -m tensor_model_transformer_tp_gb300.timeline gemm 2048 4096 1024 [epilogue]
    python -m tensor_model_transformer_tp_gb300.timeline attn_bwd 4 2048 20
    python -m tensor_model_transformer_tp_gb300.timeline attn_fwd 4 2048 20

GEMM: C[M, N] = A[M, K] B[N, K]^T in bf16 with the given epilogue (0 store,
1 bias, 2 bias + GeLU; default 2), L2 flushed by a 256 MiB write before each
launch; the CUDA-event time is the median of 20 launches, the stamps are from
one more.  Attention backward: batch x seq, heads of 128, causal; the stamps
are those of CTA 0 of the dQ (its first item) and dK/dV kernels per block,
and the span of each kernel from its first item's start (dQ) or first CTA's
entry (dK/dV) to the last end.
"""
from __future__ import annotations

import ctypes
import heapq
import sys

import numpy as np

ATTN_TIMELINE_STAMPS = 50692  # uint64 stamps in an attention timeline buffer
ATTN_FWD_STAMPS = ("entry", "set up", "Q and K_0 landed", "tile 0 saw S_0(0)",
                   "tile 0 last PV done", "tile 1 last PV done", "tile 1 O stored", "exit")
GEMM_STAMPS = {0: "entry", 1: "prologue done", 2: "first stage landed", 3: "tile 0 MMAs done",
               4: "tile 0 epilogue done", 5: "tile 1 MMAs done", 6: "tile 1 epilogue done",
               7: "tile 2 MMAs done", 8: "tile 2 epilogue done", 15: "exit"}


def _lib():
    import tensor_model_transformer_tp_gb300 as oz
    oz.build_library()
    return oz.lib()


def _median_us(torch, f, st, flush, reps=20):
    evs = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        assert f() == 0
        e1.record(st)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return float(np.median([a.elapsed_time(b) for a, b in evs])) * 1e3


def gemm(M: int, N: int, K: int, epilogue: int = 2) -> dict:
    import torch
    L = _lib()
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    L.oases_debug_gemm.argtypes = [i32, i32, i32, i32, vp, i64, i32, vp, i64, i32, i32, vp, i64,
                                   i32, vp, vp, vp, i64, i32, vp]
    L.oases_debug_gemm_timeline.argtypes = [vp]
    dev = torch.device("cuda")
    st = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    A = torch.randn(M, K, device=dev).bfloat16()
    B = (torch.randn(N, K, device=dev) * 0.02).bfloat16()
    C = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
    bias = torch.zeros(N, device=dev, dtype=torch.bfloat16)
    f = lambda: L.oases_debug_gemm(M, N, K, 1, A.data_ptr(), K, 1, B.data_ptr(), K, 1, epilogue,
                                   C.data_ptr(), N, 1, None, bias.data_ptr() if epilogue else None,
                                   None, 0, 2, st.cuda_stream)
    t = _median_us(torch, f, st, flush)
    tl = torch.zeros(16 * 4096, dtype=torch.int64, device=dev)
    assert L.oases_debug_gemm_timeline(tl.data_ptr()) == 0
    try:
        flush.zero_()
        torch.cuda.synchronize()
        assert f() == 0
        torch.cuda.synchronize()
    finally:
        assert L.oases_debug_gemm_timeline(None) == 0
    r = tl.cpu().numpy().reshape(4096, 16)
    r = r[r[:, 0] > 0]
    t0 = r[:, 0].min()
    out = {"shape": (M, N, K), "event_us": t, "ctas": len(r),
           "tflops": 2.0 * M * N * K / t / 1e6, "stamps": {}}
    for c, name in GEMM_STAMPS.items():
        v = (r[:, c][r[:, c] > 0] - t0) / 1000.0
        if len(v):
            out["stamps"][name] = (float(v.min()), float(np.median(v)), float(v.max()), len(v))
    return out


def attention_bwd(B: int, S: int, heads: int) -> dict:
    import torch
    L = _lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.oases_debug_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                        i32, vp]
    L.oases_debug_attention_timeline.argtypes = [vp]
    d = 128
    M, H = B * S, heads * d
    dev = torch.device("cuda")
    qkv = torch.randn(M, 3 * H, device=dev).bfloat16()
    o = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(heads, M, device=dev)
    do = torch.randn(M, H, device=dev).bfloat16()
    delta = torch.empty(heads, M, device=dev)
    dqkv = torch.empty(M, 3 * H, dtype=torch.bfloat16, device=dev)
    tl = torch.zeros(ATTN_TIMELINE_STAMPS, dtype=torch.int64, device=dev)

    def run(bwd):
        return L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       do.data_ptr() if bwd else None,
                                       delta.data_ptr() if bwd else None,
                                       dqkv.data_ptr() if bwd else None, B, S, heads, d, 1, 1, bwd,
                                       2 if not bwd else 0, None)
    assert run(0) == 0
    for _ in range(3):
        assert run(1) == 0
    torch.cuda.synchronize()
    assert L.oases_debug_attention_timeline(tl.data_ptr()) == 0
    try:
        assert run(1) == 0
        torch.cuda.synchronize()
    finally:
        assert L.oases_debug_attention_timeline(None) == 0
    t = tl.cpu().numpy().astype(np.int64)
    ncta = heads * B * ((S + 127) // 128)
    out = {"shape": (B, S, heads), "kernels": {}}
    for kid, name in ((1, "dq"), (2, "dkv")):
        r = t[(kid - 1) * 8192:(kid - 1) * 8192 + 2 * min(ncta, 4096)].reshape(-1, 2)
        blk = t[16384 + (kid - 1) * 256:16384 + kid * 256].reshape(64, 4)
        b0 = blk[blk > 0].min() if (blk > 0).any() else 0
        G = min(ncta, torch.cuda.get_device_properties(0).multi_processor_count)
        t0 = r[:, 0][r[:, 0] > 0].min() if (r[:, 0] > 0).any() else 0
        items0, k = [], 0  # dq: CTA 0's items in the order it ran them: start, end (us)
        while kid == 1:
            i = k * G + (G - 1 if k % 2 else 0)
            if i >= min(ncta, 4096):
                break
            items0.append((int(i), float(r[i, 0] - t0) / 1000.0, float(r[i, 1] - t0) / 1000.0))
            k += 1
        out["kernels"][name] = {
            "cta0_items": items0,
            "span_us": float(r[:, 1].max() - r[:, 0].min()) / 1000.0,
            # dq: per work item (the kernel is persistent); dK/dV: per CTA
            "cta_mean_us": float((r[:, 1] - r[:, 0]).mean()) / 1000.0,
            # per block of CTA 0: S/dP MMAs issued, accumulation MMAs issued,
            # element-wise warp 2 saw S, handed its dS (ns from the first stamp)
            "cta0_blocks_ns": [[int(x - b0) if x > 0 else -1 for x in blk[j]]
                               for j in range(64) if (blk[j] > 0).any()],
        }
    return out


def attention_fwd(B: int, S: int, heads: int) -> dict:
    """Per-item stamps of one causal forward launch (L2 flushed before it).

    An item is 256 queries of one (sequence, head); the kernel is persistent,
    so a CTA runs several items one after another."""
    import torch
    L = _lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.oases_debug_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                        i32, vp]
    L.oases_debug_attention_timeline.argtypes = [vp]
    d = 128
    M, H = B * S, heads * d
    dev = torch.device("cuda")
    st = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    qkv = torch.randn(M, 3 * H, device=dev).bfloat16()
    o = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(heads, M, device=dev)
    f = lambda: L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), None, None,
                                        None, B, S, heads, d, 1, 1, 0, 2, None)
    t = _median_us(torch, f, st, flush)
    tl = torch.zeros(ATTN_TIMELINE_STAMPS, dtype=torch.int64, device=dev)
    assert L.oases_debug_attention_timeline(tl.data_ptr()) == 0
    try:
        flush.zero_()
        torch.cuda.synchronize()
        assert f() == 0
        torch.cuda.synchronize()
    finally:
        assert L.oases_debug_attention_timeline(None) == 0
    a = tl.cpu().numpy().astype(np.int64)
    pairs = (S + 255) // 256
    items = min(heads * B * pairs, 4096)
    r = a[17920:17920 + 8 * items].reshape(items, 8)
    t0 = r[:, 0].min()
    ck = a[50688:50692]
    sm_mhz = float(ck[3] - ck[1]) / float(ck[2] - ck[0]) * 1000.0 if ck[2] > ck[0] else 0.0
    out = {"shape": (B, S, heads), "event_us": t, "items": items, "sm_mhz": sm_mhz,
           "ctas": min(heads * B * pairs, torch.cuda.get_device_properties(0).multi_processor_count),
           "span_us": float(r[:, 7].max() - t0) / 1000.0, "stamps": {}, "by_pair": []}
    for c, name in enumerate(ATTN_FWD_STAMPS):
        ok = r[:, c] > 0
        if ok.any():
            v = (r[ok, c] - r[ok, 0]) / 1000.0  # from the entry of the item's CTA
            out["stamps"][name] = (float(v.min()), float(np.median(v)), float(v.max()), int(ok.sum()))
    # the first item of CTA 0, per tile and key block: S issued, the softmax
    # saw S, the last of its four warps published P, PV ready to issue, PV
    # issued (ns from the first stamp)
    blk = a[16896:17920].reshape(2, 64, 8)
    b0 = blk[blk > 0].min() if (blk > 0).any() else 0
    out["cta0_blocks_ns"] = [[[int(x - b0) if x > 0 else -1
                               for x in (blk[t, j, 0], blk[t, j, 1], blk[t, j, 2:6].max(), blk[t, j, 7],
                                         blk[t, j, 6])]
                              for j in range(64) if (blk[t, j] > 0).any()] for t in range(2)]
    # items are numbered heaviest pair first: item i has pair pairs - 1 - i // (B heads)
    pair = pairs - 1 - np.arange(items) // (heads * B)
    # the items of the first and the last CTA in the order they ran (the
    # launch's schedule: items in index order, heaviest first, each to the
    # CTA with the least work so far, ties to the lower CTA; work = 4 x the
    # item's key blocks + 3)
    G = out["ctas"]
    nkv = (S + 127) // 128
    heap = [(0, c) for c in range(G)]
    heapq.heapify(heap)
    owner = []
    for i in range(heads * B * pairs):
        p = pairs - 1 - i // (heads * B)
        q1 = p * 256 + 128
        n1 = 0 if q1 >= S else min(q1 // 128 + 1, nkv)
        n0 = min(p * 256 // 128 + 1, nkv)
        load, c = heapq.heappop(heap)
        owner.append(c)
        heapq.heappush(heap, (load + 4 * max(n0, n1) + 3, c))
    out["cta_items"] = {}
    for c in (0, G - 1):
        out["cta_items"][c] = [(int(i), int(pair[i])) + tuple(round(float(x - t0) / 1000.0, 2) if x > 0 else -1.0
                                                             for x in r[i, 2:7])
                               for i in range(items) if owner[i] == c]
    end = np.where(r[:, 6] > 0, r[:, 6], r[:, 4])  # O stored (tile 1), else tile 0's last PV
    for p in range(pairs - 1, -1, -1):
        sel = pair == p
        if sel.any():
            out["by_pair"].append((int(p), float(np.median(end[sel] - r[sel, 2])) / 1000.0,
                                   float(np.median(r[sel, 2] - t0)) / 1000.0))
    return out


def main(argv):
    if len(argv) >= 4 and argv[0] == "gemm":
        r = gemm(int(argv[1]), int(argv[2]), int(argv[3]), int(argv[4]) if len(argv) > 4 else 2)
        print("%dx%dx%d: %.1f us (CUDA events), %.0f TFLOP/s, %d CTAs" % (*r["shape"], r["event_us"],
                                                                      r["tflops"], r["ctas"]))
        for name, (lo, med, hi, n) in r["stamps"].items():
            print("  %-22s min %6.2f  median %6.2f  max %6.2f us  (%d CTAs)" % (name, lo, med, hi, n))
    elif len(argv) == 4 and argv[0] == "attn_fwd":
        r = attention_fwd(int(argv[1]), int(argv[2]), int(argv[3]))
        print("attention forward %dx%dx%d: %.1f us (CUDA events), span %.1f us, %d items, "
              "SM clock %.0f MHz (CTA 0)" % (*r["shape"], r["event_us"], r["span_us"], r["items"],
                                             r["sm_mhz"]))
        for name, (lo, med, hi, n) in r["stamps"].items():
            print("  %-22s min %6.2f  median %6.2f  max %6.2f us after its CTA's entry (%d items)"
                  % (name, lo, med, hi, n))
        for p, life, start in r["by_pair"]:
            print("  tile pair %2d: median item time %6.2f us (Q_0, K_0 landed to O stored), "
                  "median start %6.2f us" % (p, life, start))
        for c, rows in r["cta_items"].items():
            print("  CTA %d items (us from the kernel's first entry): item, pair, Q_0/K_0 landed, "
                  "tile 0 saw S_0(0), tile 0 / tile 1 last PV done, tile 1 O stored" % c)
            for row in rows:
                print("    %4d %2d  %s" % (row[0], row[1], " ".join("%7.2f" % x for x in row[2:])))
        print("  CTA 0, first item, per block (ns): S issued, softmax saw S, P published, PV ready, "
              "PV issued")
        for t in range(2):
            for j, row in enumerate(r["cta0_blocks_ns"][t][:8]):
                print("  tile %d block %2d: %s" % (t, j, " ".join("%7d" % x for x in row)))
    elif len(argv) == 4 and argv[0] == "attn_bwd":
        r = attention_bwd(int(argv[1]), int(argv[2]), int(argv[3]))
        for name, k in r["kernels"].items():
            print("%s: span %.1f us, %s mean %.1f us" % (name, k["span_us"],
                                                         "item" if name == "dq" else "CTA",
                                                         k["cta_mean_us"]))
            if k["cta0_items"]:
                print("  CTA 0 items (us): " + ", ".join("%d: %.1f-%.1f" % x for x in k["cta0_items"]))
            print("  CTA 0 per block (ns): SdP issued, ACC issued, warp 2 saw S, warp 2 handed dS")
            for j, row in enumerate(k["cta0_blocks_ns"][:8]):
                print("  block %d: %s" % (j, " ".join("%6d" % x for x in row)))
    else:
        print(__doc__)
        return 2
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
