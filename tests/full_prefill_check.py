"""The 16K-token prefill layer (Edge0 shape, Zipf router bias) against the
oracle on EVERY token, not a sample: routing (logits within the bar, expert
sets bit-exact on unambiguous tokens, weights) and the bf16 outputs of every
unambiguous token. Too slow for the test suite (the fp64 oracle needs tens
of core-minutes), so it runs as a script and prints one summary line:

    python tests/full_prefill_check.py [--workload prefill_t16384_zipf] [--procs N]

The oracle runs in a process pool made before the first CUDA call (forked
workers share the generated weights), in chunks of tokens, while the GPU
computes the layer.
"""
import argparse
import multiprocessing as mp
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import lmoe_synth as S  # noqa: E402
import oracle as O  # noqa: E402

_W = {}


def _oracle_chunk(bounds):
    a, b = bounds
    sh, W, x = _W["sh"], _W["W"], _W["x"]
    y, idx, w, lg = O.layer_forward(O.Layer(sh, W), x[a:b])
    return a, y, idx, w, lg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="prefill_t16384_zipf")
    ap.add_argument("--procs", type=int, default=0, help="oracle processes (0: every host core)")
    ap.add_argument("--chunk", type=int, default=64)
    args = ap.parse_args()

    sh, T, W, x = S.make_workload(args.workload)
    _W.update(sh=sh, W=W, x=x)
    O.build()
    procs = args.procs or os.cpu_count() or 1
    t0 = time.time()
    # forked before any CUDA call: the workers share W and x and never touch the GPU
    pool = mp.get_context("fork").Pool(procs)
    chunks = [(a, min(T, a + args.chunk)) for a in range(0, T, args.chunk)]
    pending = pool.map_async(_oracle_chunk, chunks)

    import torch
    from gpu_util import bf16_bits, bf16_tensor, check_outputs, check_routing
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    dev = torch.device("cuda:0")
    m = LatentMoE(sh, W, device=0, force_path=capi.PATH_AUTO)
    assert capi.lmoe_stage_name(m.h, T, 1)[0] == "permute", "the prefill path must run"
    xt = bf16_tensor(x, dev)
    idx, w, lg = m.route(xt, want_logits=True)
    y = bf16_bits(m.forward(xt))
    torch.cuda.synchronize()
    m.check()
    idx_g, w_g, lg_g = idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()
    t_gpu = time.time() - t0

    y_ref = np.empty((T, sh.d))
    idx_ref = np.empty((T, sh.k), np.int32)
    w_ref = np.empty((T, sh.k))
    lg_ref = np.empty((T, sh.E))
    for a, yy, ii, ww, ll in pending.get():
        n = yy.shape[0]
        y_ref[a:a + n], idx_ref[a:a + n], w_ref[a:a + n], lg_ref[a:a + n] = yy, ii, ww, ll
    pool.close()
    pool.join()
    t_all = time.time() - t0

    keep = check_routing(lg_g, idx_g, w_g, lg_ref, idx_ref, w_ref, sh.k)
    mr, ma, _ = check_outputs(y[keep], y_ref[keep], f"{args.workload}, every token")
    lerr = (np.abs(lg_g.astype(np.float64) - lg_ref).max(axis=1) / np.abs(lg_ref).max(axis=1)).max()
    print(f"{args.workload}: all {T} tokens against the oracle ({procs} oracle processes, {t_all:.0f} s; "
          f"GPU done at {t_gpu:.0f} s): logits worst {lerr:.2e} of max|l| (bar 1e-5), expert sets "
          f"identical on {int(keep.sum())} unambiguous tokens ({int((~keep).sum())} near-tie tokens "
          f"excluded), outputs mean rel {mr:.2e} (bar 1e-3), max abs {ma:.2e} (bar 2e-2): PASS", flush=True)


if __name__ == "__main__":
    main()
