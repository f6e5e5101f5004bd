"""Small builders for hand-made instances used by the pin tests."""
import numpy as np

from memory_aware_device_gb300.synth import Instance

BIG = 1 << 60


def make(L=1, fl=0, pd=0, pe=0, ao=0, aw=0, a2a=0, moe=0, G=(8,), bw=(1000,), lat=(0,),
         cand=(0,), strat=((1, 1, 1, 0, 0),), D=8, unit=1, Pmax=1, R=1, M=1, budget=BIG,
         opt=6):
    def col(v, dt=np.int64):
        a = np.asarray(v, dtype=dt)
        return np.full(L, a, dtype=dt) if a.ndim == 0 else a
    return Instance(L=L, D=D, unit=unit, Pmax=Pmax, R=R, M=M, budget=budget, opt_factor=opt,
                    fl=col(fl), pd=col(pd), pe=col(pe), ao=col(ao), aw=col(aw), a2a=col(a2a),
                    moe=col(moe, np.uint8), tierG=np.asarray(G, np.int64),
                    tierBw=np.asarray(bw, np.int64), tierLat=np.asarray(lat, np.int64),
                    cand=np.asarray(cand, np.int32),
                    strat=np.asarray(strat, np.int16).reshape(-1, 5))


def log2(k):
    return int(k).bit_length() - 1
