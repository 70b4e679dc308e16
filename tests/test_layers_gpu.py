"""One decoder layer (GPU, through clef_decoder_layer) against the oracle's fp64 layer.

Full-size cases of the target: a Gated DeltaNet layer at L = 1024 and a gated full-attention
layer at L = 4096, batch 1, with seeded random LUT-6 weights and fp16 N(0, 1) inputs.  The bound
is the target's per-layer 5e-3 relative RMSE on the layer output; the change the layer makes
(output - input) is reported and held to 1e-2.
"""
import numpy as np
import pytest

import synth
from oracle import model as om
from tests._util import min_row_cosine, rel_rmse

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
from full_attention_prefill_gb300.model import ATTENTION, GDN, DeviceLayer  # noqa: E402

LAYER_TOL = 5e-3
DELTA_TOL = 1e-2


def run_layer(layer_index, L, B=1, seed=0):
    w = synth.layer_weights(seed, layer_index)
    attention = synth.is_attention_layer(layer_index)
    dl = DeviceLayer(w, ATTENTION if attention else GDN)
    x = synth.normal_f16(seed, "layer.x", layer_index * 100 + B, (B, L, 4096))
    xd = torch.from_numpy(x.astype(np.float32)).cuda()
    clef.decoder_layer(dl, xd)
    clef.sync_status()
    y = xd.double().cpu().numpy()
    for b in range(B):
        ref = om.decoder_layer(x[b], w, attention)
        e_out = rel_rmse(y[b], ref)
        e_delta = rel_rmse(y[b] - x[b], ref - x[b])
        cos = min_row_cosine(y[b] - x[b], ref - x[b])
        print(f"layer {layer_index} L={L} b={b}: out rel-RMSE {e_out:.2e}, delta rel-RMSE "
              f"{e_delta:.2e}, min row cos {cos:.6f}")
        assert e_out < LAYER_TOL
        assert e_delta < DELTA_TOL


# (4096, 1): the scan runs in pieces on two streams, with the z-gated norm per piece;
# (9856, 1): 77 token tiles of 128, so the a/b projection runs without a K split and writes the
# gates from its own epilogue (shorter inputs split K and sum the parts in a second kernel)
@pytest.mark.parametrize("L,B", [(1024, 1), (70, 2), (4096, 1), (9856, 1)])
def test_gdn_layer(L, B):
    run_layer(0, L, B)


@pytest.mark.parametrize("L,B", [(4096, 1), (70, 2)])
def test_attention_layer(L, B):
    run_layer(3, L, B)
