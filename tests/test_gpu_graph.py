"""decode_step under CUDA-graph capture: one serving step over three layers
(append of the current token + attention, per layer) captured into a graph and
replayed must write the same cache bytes, outputs and lse as the same calls
run eagerly, and replaying it again (same positions, same inputs) must leave
them unchanged.  The step's launches use programmatic dependent launch and, at
head_dim 256/512, a thread-block cluster; both must survive capture.  Cases
cover G = 8 with the separate V un-rotation kernel and the Lloyd-Max, K-only
INT2 and in-quant Hadamard modes."""
import numpy as np
import pytest
import torch

from int2_kv_cache_append_gb300 import oscar_kv as K
from int2_kv_cache_append_gb300 import synth as S

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs CUDA")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int2_kv_cache_append_gb300 import build
    build.build()


@pytest.mark.parametrize("D,B,Hq,Hkv,flags", [
    (128, 4, 16, 4, 0),
    (256, 2, 8, 2, 0),
    (512, 2, 16, 2, 0),                     # G = 8, V un-rotated by unrot_kernel
    (128, 2, 16, 2, K.FLAG_LLOYD_MAX),
    (128, 2, 8, 2, K.FLAG_V_BF16),
    (128, 2, 8, 2, K.FLAG_HADAMARD | K.FLAG_ABSORB_V),
])
def test_graph_replay_equals_eager(D, B, Hq, Hkv, flags):
    L, S_, W, cap = 3, 16, 64, 1500
    kc = K.KVConfig(L, B, Hq, Hkv, D, S_, W, cap, 0.96, 0.92, K.FLAG_OUT_FP32 | flags)
    lay = K.layout_query(kc)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77 + D)
    ch = np.array([3, 40])
    rng = np.random.default_rng(D)
    if flags & K.FLAG_HADAMARD:
        rots = [(None, None)] * L
    else:
        rots = [(torch.from_numpy(S.qr_rotation(rng, D).astype(np.float32)).cuda(),
                 torch.from_numpy(S.qr_rotation(rng, D).astype(np.float32)).cuda()) for _ in range(L)]
    cache0 = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device="cuda")
    T0 = 1200
    for layer in range(L):
        K.kv_append(kc, cache0, layer, S.activations_torch(gen, (B, T0, Hkv, D), ch, dtype=torch.bfloat16),
                    S.activations_torch(gen, (B, T0, Hkv, D), ch, dtype=torch.bfloat16),
                    torch.zeros(B, dtype=torch.int32, device="cuda"), *rots[layer])
    k1 = S.activations_torch(gen, (B, 1, Hkv, D), ch, dtype=torch.bfloat16)
    v1 = S.activations_torch(gen, (B, 1, Hkv, D), ch, dtype=torch.bfloat16)
    q = S.activations_torch(gen, (B, Hq, D), ch, dtype=torch.bfloat16)
    start = torch.full((B,), T0, dtype=torch.int32, device="cuda")
    seq = start + 1
    ws = torch.empty(lay["decode_workspace_bytes"], dtype=torch.uint8, device="cuda")

    def run(cache, outs, lses, st):
        for layer in range(L):
            K.decode_step(kc, cache, layer, k1, v1, start, q, seq, *rots[layer], outs[layer], ws, lse=lses[layer],
                          seq_len_hint=cap, status=st)

    def buffers():
        return ([torch.full((B, Hq, D), float("nan"), device="cuda") for _ in range(L)],
                [torch.full((B, Hq), float("nan"), device="cuda") for _ in range(L)],
                torch.zeros(1, dtype=torch.int32, device="cuda"))

    # eager
    ce = cache0.clone()
    oe, le, se = buffers()
    run(ce, oe, le, se)
    torch.cuda.synchronize()
    # captured on a side stream, then replayed
    cg = cache0.clone()
    og, lg, sg = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run(cg, og, lg, sg)
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(3):
        graph.replay()
        torch.cuda.synchronize()
        assert int(se.item()) == int(sg.item()) == 0
        assert torch.equal(ce, cg), f"cache differs after replay {rep}"
        for layer in range(L):
            assert torch.equal(oe[layer], og[layer]), f"layer {layer} output differs after replay {rep}"
            assert torch.equal(le[layer], lg[layer]), f"layer {layer} lse differs after replay {rep}"
