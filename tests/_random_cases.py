"""Seeded random problem configurations for the randomized oracle and GPU
parity tests: every mode (SWA / CSA / HCA / token-wise top-k), layout pair,
dtype, head count, window, mask mode, block size, packed format, block-wise
selection and row padding the parameter rules allow, at sizes the oracle and
the brute force finish in well under a second."""
import numpy as np

MODES = ("swa", "csa", "hca", "ori_sparse")


def random_case(seed: int):
    rng = np.random.default_rng(7919 * seed + 17)
    mode = MODES[seed % len(MODES)]
    layout_q = str(rng.choice(["BSND", "TND"]))
    layout_kv = str(rng.choice([layout_q, "PAGED"]))
    B = int(rng.integers(1, 4))
    kw = dict(mode=mode, layout_q=layout_q, layout_kv=layout_kv, dtype=str(rng.choice(["bf16", "fp16"])),
              sinks=bool(rng.random() < 0.5))
    if layout_q == "BSND":
        q_s = int(rng.integers(1, 4))
        kw["q_lens"] = [q_s] * B
        if rng.random() < 0.3:
            kw["seqused_q"] = [int(x) for x in rng.integers(1, q_s + 1, B)]
    else:
        kw["q_lens"] = [int(x) for x in rng.integers(1, 5, B)]
    kw["kv_lens"] = [int(x) for x in rng.integers(1, 400, B)]
    q_n = int(rng.choice([1, 3, 8, 16, 40, 64, 96, 128]))
    if layout_kv == "PAGED":
        kw["ori_block_size"] = int(rng.choice([16, 32, 48, 64, 128]))
        kw["cmp_block_size"] = int(rng.choice([16, 32, 80]))
    if mode != "ori_sparse":
        kw["win_left"] = int(rng.choice([-1, 0, 3, 17, 127]))
        kw["win_right"] = int(rng.choice([-1, 0, 0, 2]))
        kw["ori_mask_mode"] = int(rng.choice([4, 4, 3, 0]))
        if rng.random() < 0.25:
            kw["kv_row_pad"] = 48
    if mode == "csa":
        kw["cmp_ratio"] = int(rng.choice([2, 4]))
        kw["cmp_topk"] = int(rng.choice([4, 8, 16, 32]))
        kw["index_mode"] = str(rng.choice(["visible", "visible", "any"]))
    elif mode == "hca":
        kw["cmp_ratio"] = int(rng.choice([4, 8, 16]))
        kw["cmp_mask_mode"] = int(rng.choice([3, 3, 0]))
    elif mode == "ori_sparse":
        fmt = str(rng.choice(["plain", "int8_packed", "fp8_packed"]))
        kw["kv_format"] = fmt
        kw["ori_topk"] = int(rng.integers(2, 20))
        kw["index_mode"] = str(rng.choice(["visible", "any"]))
        if fmt != "plain":
            kw["rope_head_dim"] = int(rng.choice([0, 64]))
        kw["sparse_block_size"] = int(rng.choice([1, 1, 2, 4, 16]))
    return f"random{seed}_{mode}", q_n, kw


SEEDS = list(range(48))
