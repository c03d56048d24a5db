"""Writes the router biases that give the Zipf-shaped expert loads.

Usage:  python -m oracle.calibrate_zipf [workload ...]     (default: all "zipf" workloads)

Calls only the oracle (f64) and the seeded generator.  For each workload with
bias == "zipf" it writes synth/zipf_bias_<name>.txt, which the tests and the
benchmark read as an input.

Procedure (the pages say expert popularity is Zipf-like -- pure-C Colibri
tutorial, trdm.cn, §2.1 -- but give no recipe, so this one is ours):
  * target share p_e proportional to rank_e^-s over a seeded expert
    permutation, water-filled so no share exceeds 1/k (a token selects an
    expert at most once, so an expert can hold at most 1/k of assignments);
  * a calibration batch of 4096 tokens drawn with its own seed;
  * 128 fixed iterations of
        b_e += 0.5 * 0.97^i * spread * clip(ln target_e - ln observed_e, -1, 1),
    where observed_e is the expert's share of the batch's assignments (floored
    at half an assignment) and spread is the standard deviation of the
    bias-free selection key over the batch (the logit z for softmax routers,
    sigmoid(z) for sigmoid routers), so the step is in the key's own units;
  * the bias is a softmax logit offset (softmax routers) or the noaux_tc
    selection bias (sigmoid routers).
"""
import hashlib
import os
import sys

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

CAL_TOKENS = 4096
ITERS = 128
CAL_SEED_XOR = 0xCA11B8A7E


def zipf_target(wl):
    E, k, s = wl.E, wl.k, wl.zipf_s
    keys = [synth.draw(wl.seed, 0, synth.T_BIAS, 0x5A1F, e) for e in range(E)]
    order = np.argsort(np.array(keys, dtype=np.uint64), kind="stable")
    rank = np.empty(E, np.int64)
    rank[order] = np.arange(1, E + 1)
    p = rank.astype(np.float64) ** (-s)
    p /= p.sum()
    cap = 1.0 / k
    capped = np.zeros(E, bool)
    while True:
        over = (p > cap + 1e-15) & ~capped
        if not over.any():
            break
        capped |= over
        free_mass = 1.0 - cap * capped.sum()
        rest = ~capped
        p[capped] = cap
        p[rest] = p[rest] / p[rest].sum() * free_mass
    return p


def calibrate(wl, verbose=True):
    L = oracle.layout(wl)
    Wr = synth.router_w(wl)
    cal_seed = wl.seed ^ CAL_SEED_XOR
    fill = synth.normal_bf16 if wl.x_dtype == synth.workloads.X_BF16 else synth.normal_f32
    x = fill(cal_seed, 0, synth.T_X, 0, CAL_TOKENS * wl.H, 1.0).reshape(CAL_TOKENS, wl.H)
    W = oracle.weights(L, Wr, None)
    z = oracle.router_logits(L, W, x)
    target = zipf_target(wl)
    A = CAL_TOKENS * wl.k
    base = z if wl.router_mode == synth.workloads.ROUTER_SOFTMAX else 1.0 / (1.0 + np.exp(-z))
    spread = float(base.std())
    b = np.zeros(wl.E, np.float64)
    for i in range(ITERS):
        idx, _, _, _ = oracle.route_from_logits(L, b.astype(np.float32), z)
        obs = np.bincount(idx.ravel(), minlength=wl.E).astype(np.float64)
        obs = np.maximum(obs, 0.5) / A
        b += 0.5 * 0.97 ** i * spread * np.clip(np.log(target) - np.log(obs), -1.0, 1.0)
    b32 = b.astype(np.float32)
    idx, _, _, _ = oracle.route_from_logits(L, b32, z)
    load = np.bincount(idx.ravel(), minlength=wl.E)
    stats = dict(max_load=int(load.max()), cv=float(load.std() / load.mean()),
                 empty=int((load == 0).sum()))
    digest = hashlib.sha256(b32.tobytes()).hexdigest()[:16]
    if verbose:
        print("%s: max load %d of %d tokens, cv %.3f, empty experts %d, sha256[:16] %s"
              % (wl.name, stats["max_load"], CAL_TOKENS, stats["cv"], stats["empty"], digest))
    return b32, stats, digest


def write(wl, b32, stats, digest):
    path = synth.zipf_bias_path(wl)
    with open(path, "w") as f:
        f.write("# router bias for workload %s: Zipf(s=%.2f) expert loads, E=%d, k=%d\n"
                % (wl.name, wl.zipf_s, wl.E, wl.k))
        f.write("# written by oracle/calibrate_zipf.py (oracle f64 routing, %d-token calibration "
                "batch, %d iterations)\n" % (CAL_TOKENS, ITERS))
        f.write("# calibration batch: max load %d, cv %.3f, empty experts %d; sha256(f32)[:16] %s\n"
                % (stats["max_load"], stats["cv"], stats["empty"], digest))
        for v in b32:
            f.write("%.9g\n" % float(v))
    return path


def main(names):
    wls = [synth.BY_NAME[n] for n in names] if names else [w for w in synth.ALL if w.bias == "zipf"]
    for wl in wls:
        b32, stats, digest = calibrate(wl)
        print("wrote", write(wl, b32, stats, digest))


if __name__ == "__main__":
    main(sys.argv[1:])
