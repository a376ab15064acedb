"""Shared helpers of the GPU parity tests: run the CUDA path through the binding and
the oracle on the same seeded inputs, and map padded GPU rows to the oracle's
compact rows."""
import numpy as np
import torch

import oracle


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def inputs_np(inp):
    return (inp.x.double().numpy(), inp.logits.numpy(), inp.w_gu.float().numpy(),
            inp.w_down.float().numpy(), None if inp.dy is None else inp.dy.double().numpy())


def row_maps(counts: np.ndarray, padded: np.ndarray, offsets: np.ndarray):
    """(gpu_rows, oracle_rows): the same dispatched rows in the padded and compact spaces."""
    g, o = [], []
    for e, c in enumerate(counts):
        g.append(padded[e] + np.arange(c))
        o.append(offsets[e] + np.arange(c))
    return np.concatenate(g).astype(np.int64), np.concatenate(o).astype(np.int64)


def check_dispatch_exact(views: dict, ref: dict, x_bf16: torch.Tensor, k: int) -> None:
    """Bit-exact comparison of counts, offsets, the permutation and the row copies."""
    counts = to_np(views["counts"]).astype(np.int64)
    offsets = to_np(views["offsets"]).astype(np.int64)
    padded = to_np(views["padded_offsets"]).astype(np.int64)
    assert np.array_equal(counts, ref["counts"]), "expert counts differ"
    assert np.array_equal(offsets, ref["offsets"]), "compact offsets differ"
    want_pad = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    assert np.array_equal(padded, want_pad), "padded offsets differ from their definition"
    ids = ref["ids"].astype(np.int64)
    row_of = to_np(views["row_of"]).astype(np.int64)
    rank_gpu = row_of - padded[ids]
    rank_ref = ref["row_of"] - ref["offsets"][ids]
    assert np.array_equal(rank_gpu, rank_ref), "permutation order differs"
    tok_of = to_np(views["tok_of"]).astype(np.int64)
    grow, orow = row_maps(counts, padded, offsets)
    assert np.array_equal(tok_of[grow], ref["tok_of"][orow]), "tok_of differs"
    pad_mask = np.ones(int(padded[-1]), dtype=bool)
    pad_mask[grow] = False
    assert (tok_of[:int(padded[-1])][pad_mask] == -1).all(), "padding rows must hold -1"
    xp = views["xp"]
    tok = torch.from_numpy(ref["tok_of"][orow])
    assert torch.equal(xp[torch.from_numpy(grow).to(xp.device)].cpu(), x_bf16[tok]), \
        "dispatched rows are not exact copies"
    if pad_mask.any():
        assert not xp[:int(padded[-1])][torch.from_numpy(pad_mask).to(xp.device)].any(), \
            "padding rows of xp must be zero"
