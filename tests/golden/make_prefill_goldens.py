"""Write the stored expected rows of the full-size prefills, computed by the oracle alone.

    python tests/golden/make_prefill_goldens.py [--only l16384|b32x512]

Two workloads, the seeded synthetic model (weights seed 0, token ids of seed 1000, the ids of the
first request of the throughput bench):
  * one request of 16,384 positions through all 32 layers: the final-norm hidden rows at
    `L16384_ROWS` -> prefill_l16384_rows.npz;
  * requests 0, 13 and 31 of the 32 requests of 512 positions (ids seed 1000, one [32, 512]
    draw): the rows at `B32_ROWS` of each -> prefill_b32x512_rows.npz.
Each file holds the positions, the rows (float32 of the oracle's float64 result), the seeds and
the number of oracle threads.  Nothing here reads the CUDA library: the inputs come from
synth/, the values from oracle/ (the 16,384-position prefill takes about 1.5 h on 8 cores).
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import _lib, model  # noqa: E402

WEIGHT_SEED = 0
IDS_SEED = 1000
# positions: both ends, every 64-position chunk edge of interest and every 4,096-position edge,
# plus a spread of others (sorted, unique)
L16384_ROWS = sorted({0, 1, 63, 64, 127, 128, 511, 512, 1023, 2047, 2048, 4095, 4096, 4097, 6000,
                      8191, 8192, 8193, 10000, 12287, 12288, 14000, 16000, 16320, 16382, 16383}
                     | set(range(301, 16383, 1789)))
B32_REQUESTS = (0, 13, 31)
B32_ROWS = (0, 1, 63, 64, 255, 256, 400, 511)


def _prefill(ids):
    emb = synth.embedding_rows(WEIGHT_SEED, ids)
    return model.prefill(ids, emb, lambda l: synth.layer_weights(WEIGHT_SEED, l),
                         synth.final_norm_weight(WEIGHT_SEED), n_layers=32)


def make_l16384():
    ids = synth.token_ids(IDS_SEED, 1, 16384)[0]
    t0 = time.time()
    hidden = _prefill(ids)
    rows = np.asarray(L16384_ROWS, dtype=np.int64)
    out = os.path.join(HERE, "prefill_l16384_rows.npz")
    np.savez(out, positions=rows, rows=hidden[rows].astype(np.float32), weight_seed=WEIGHT_SEED,
             ids_seed=IDS_SEED, seconds=time.time() - t0, threads=_lib.lib().orc_num_threads())
    print(f"wrote {out} ({time.time() - t0:.0f} s)", flush=True)


def make_b32x512():
    ids = synth.token_ids(IDS_SEED, 32, 512)
    t0 = time.time()
    rows = np.asarray(B32_ROWS, dtype=np.int64)
    got = np.stack([_prefill(ids[r])[rows].astype(np.float32) for r in B32_REQUESTS])
    out = os.path.join(HERE, "prefill_b32x512_rows.npz")
    np.savez(out, requests=np.asarray(B32_REQUESTS, dtype=np.int64), positions=rows, rows=got,
             weight_seed=WEIGHT_SEED, ids_seed=IDS_SEED, seconds=time.time() - t0,
             threads=_lib.lib().orc_num_threads())
    print(f"wrote {out} ({time.time() - t0:.0f} s)", flush=True)


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", choices=["l16384", "b32x512"], default=None)
    a = ap.parse_args()
    if a.only in (None, "b32x512"):
        make_b32x512()
    if a.only in (None, "l16384"):
        make_l16384()
