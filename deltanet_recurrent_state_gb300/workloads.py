"""The five seeded synthetic workloads of the DeltaNet verify / commit / prefill path.

Shapes follow the serving setups the pages describe: one user verifying a
16-wide block (7 model drafts + 8 context drafts + 1; "HyperQwen on one RTX 3090:
a first-time developer's guide ...", What actually became faster?), the plain
7-draft decode loop, batch mode at 64 concurrent requests with 16-bit state
("HyperQwen" README, The numbers behind that), and prefix-cache checkpointing of
a ~25,000-token prompt ("HyperQwen: 1,000 tok/s on a Single RTX 3090 ...",
Technical Insight). The model geometry (48 DeltaNet layers x 48 heads x 128 x 128)
is a stated choice: the pages give none.
"""

WORKLOADS = {
    # tiny case the oracle finishes in well under a second
    "tiny_h4_d64_t8_f32": dict(
        L=1, B=1, H=4, dk=64, dv=64, T=8, io="f32", state="f32",
        V=512, logit_dtype="f32", logit_std=1.0, accept="uniform", seed=1000),
    # single user, 16-wide verify block, 15 of 16 accepted
    "single_user_l48_h48_d128_t16_f16": dict(
        L=48, B=1, H=48, dk=128, dv=128, T=16, io="f16", state="f16",
        V=151936, logit_dtype="f16", logit_std=2.0, accept="fixed", accept_value=15, seed=1001),
    # single user, 8-wide block, 1000 verify -> accept -> commit steps
    "decode_loop_l48_h48_d128_t8_f16": dict(
        L=48, B=1, H=48, dk=128, dv=128, T=8, io="f16", state="f16",
        V=151936, logit_dtype="f16", logit_std=2.0, accept="geometric", steps=1000, seed=1002),
    # batch mode: 64 requests, 4-wide blocks
    "batch64_l48_h48_d128_t4_f16": dict(
        L=48, B=64, H=48, dk=128, dv=128, T=4, io="f16", state="f16",
        V=151936, logit_dtype="f16", logit_std=2.0, accept="uniform", seed=1003),
    # one 25,000-token prompt, checkpoint every 64 tokens
    "prefill_p25000_l48_h48_d128_c64_f16": dict(
        L=48, B=1, H=48, dk=128, dv=128, P=25000, chunk=64, io="f16", state="f16", seed=1004),
}

HEADLINE = "single_user_l48_h48_d128_t16_f16"
