"""One product, repeated a few times, for profiler captures of a single kernel.

    python -m gguf_block_quantized_gb300.profile_case --case gemv_q6k_lm_head --reps 3

Cases (synthetic weights ~N(0, 0.02), activations ~N(0, 1)):
  gemv_q6k_lm_head   Q6_K 128256 x 2048, 1 token    (216 MB of weights: larger than L2)
  gemv_q6k_lm_head_4tok  the same, 4 tokens
  gemv_q4k_wide      Q4_K 32768 x 8192, 1 token     (151 MB)
  gemv_q8_0_wide     Q8_0 16384 x 8192, 1 token     (143 MB)
  gemm_q4k_ffn_up    Q4_K 14336 x 4096, 512 tokens  (prefill, tensor cores)
  gemm_q4k_ffn_down  Q4_K 4096 x 14336, 512 tokens
  gemv_llama1b_layer the seven decode products of a Llama-1B-shaped layer, one grouped call
  gemv_llama8b_layers  the grouped decode calls of two Llama-8B Q4_K_M layers, alternating:
                     layer 0 (Q6_K attn_v / ffn_down) and layer 4 (all Q4_K), the weights and
                     inputs of the benchmark's sweep
  prefill_llama8b_layer  one Llama-8B layer at 2048 tokens as a model calls it: q/k/v grouped
                     on one input, o, gate/up grouped on one input, down (Q4_K, Q6_K v/down)
"""
from __future__ import annotations

import argparse

CASES = {
    "gemv_q6k_lm_head": (3, 128256, 2048, 1),
    "gemv_q6k_lm_head_4tok": (3, 128256, 2048, 4),
    "gemv_q4k_wide": (2, 32768, 8192, 1),
    "gemv_q8_0_wide": (1, 16384, 8192, 1),
    "gemm_q4k_ffn_up": (2, 14336, 4096, 512),
    "gemm_q4k_ffn_down": (2, 4096, 14336, 512),
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", required=True, choices=sorted(CASES) + ["gemv_llama1b_layer", "gemv_llama8b_layers",
                                                                     "prefill_llama8b_layer"])
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    import torch

    from gguf_block_quantized_gb300 import syn, synth

    if args.case == "gemv_llama1b_layer":
        from gguf_block_quantized_gb300 import workloads
        mats = workloads.LLAMA1B_LAYER
        Ws = [syn.quantize(m.wtype, torch.from_numpy(synth.weight(2, i, m.n_out, m.n_in)).cuda()) for i, m in enumerate(mats)]
        Xs = [torch.from_numpy(synth.activations(2, i, 1, m.n_in)).cuda() for i, m in enumerate(mats)]
        Ys = [torch.empty((1, m.n_out), device="cuda") for m in mats]
        for _ in range(args.reps):
            syn.mul_mat_batch([(m.wtype, Ws[i], m.n_out, m.n_in, Xs[i], Ys[i]) for i, m in enumerate(mats)], 1)
        torch.cuda.synchronize()
        assert syn.device_status() == syn.OK
        print(f"{args.case}: {args.reps} grouped calls done")
        return
    if args.case == "gemv_llama8b_layers":
        from gguf_block_quantized_gb300 import workloads
        mats = workloads.llama8b_q4_k_m()
        d, f = mats[0].n_in, mats[6].n_in
        xs = [torch.from_numpy(synth.activations(5, j, 1, n)).cuda() for j, n in enumerate([d, d, d, f])]
        src = [xs[0], xs[0], xs[0], xs[1], xs[2], xs[2], xs[3]]
        calls = []
        for k in (0, 4):
            lay = mats[7 * k:7 * k + 7]
            Ws = [syn.quantize(m.wtype, torch.from_numpy(synth.weight(5, 7 * k + i, m.n_out, m.n_in)).cuda())
                  for i, m in enumerate(lay)]
            Ys = [torch.empty((1, m.n_out), device="cuda") for m in lay]
            calls.append([(m.wtype, Ws[i], m.n_out, m.n_in, src[i], Ys[i]) for i, m in enumerate(lay)])
        for _ in range(args.reps):
            for c in calls:
                syn.mul_mat_batch(c, 1)
        torch.cuda.synchronize()
        assert syn.device_status() == syn.OK
        print(f"{args.case}: {args.reps} x 2 grouped calls done")
        return
    if args.case == "prefill_llama8b_layer":
        from gguf_block_quantized_gb300 import workloads
        lay = workloads.llama8b_q4_k_m(n_layers=1, lm_head=False)  # a Q6_K attn_v / ffn_down layer
        n_tok = 2048
        Ws = [syn.quantize(m.wtype, torch.from_numpy(synth.normal(20 + i, (m.n_out, m.n_in), 0.02)).cuda())
              for i, m in enumerate(lay)]
        XA, XO, XF = (torch.from_numpy(synth.normal(30 + i, (n_tok, lay[0].n_in))).cuda() for i in range(3))
        XD = torch.from_numpy(synth.normal(33, (n_tok, lay[6].n_in))).cuda()
        Ys = [torch.empty((n_tok, m.n_out), device="cuda") for m in lay]
        syn.syn_reserve(lay[6].n_in, n_tok, torch.cuda.current_stream().cuda_stream)
        for _ in range(args.reps):
            syn.mul_mat_batch([(lay[i].wtype, Ws[i], lay[i].n_out, lay[i].n_in, XA, Ys[i]) for i in range(3)], n_tok)
            syn.mul_mat(lay[3].wtype, Ws[3], lay[3].n_out, lay[3].n_in, XO, Y=Ys[3])
            syn.mul_mat_batch([(lay[i].wtype, Ws[i], lay[i].n_out, lay[i].n_in, XF, Ys[i]) for i in (4, 5)], n_tok)
            syn.mul_mat(lay[6].wtype, Ws[6], lay[6].n_out, lay[6].n_in, XD, Y=Ys[6])
        torch.cuda.synchronize()
        assert syn.device_status() == syn.OK
        print(f"{args.case}: {args.reps} layer passes done")
        return
    wt, n_out, n_in, n_tok = CASES[args.case]
    W = syn.quantize(wt, torch.from_numpy(synth.normal(5, (n_out, n_in), 0.02)).cuda())
    X = torch.from_numpy(synth.normal(6, (n_tok, n_in))).cuda()
    Y = torch.empty((n_tok, n_out), device="cuda")
    syn.syn_reserve(n_in, n_tok, torch.cuda.current_stream().cuda_stream)
    for _ in range(args.reps):
        syn.mul_mat(wt, W, n_out, n_in, X, Y=Y)
    torch.cuda.synchronize()
    assert syn.device_status() == syn.OK
    print(f"{args.case}: {args.reps} products done")


if __name__ == "__main__":
    main()
