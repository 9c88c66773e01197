"""Work item of the parallel oracle runs in the parity tests: one head's
oracle profile and decode.  Kept free of torch and CUDA so that spawned
worker processes start quickly and never touch the GPU."""
from oracle import fastgen_oracle as O
from synth import punct_ids, special_ids


def oracle_job(job):
    Qa, Ka, Va, ids, n, steps, T, r_l, r_f, long_prompt = job
    prof = O.profile_head_long if long_prompt else O.profile_head
    r = prof(Qa[:n], Ka[:n], ids, special_ids(), punct_ids(), T, r_l, r_f)
    out, pos = O.decode_head(r["policy"], r["keep"], n, r["w"], ids, Qa, Ka, Va, special_ids(),
                             punct_ids(), steps)
    r["out"], r["final_pos"] = out, pos
    r.pop("A", None)
    return r
