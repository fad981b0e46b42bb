"""Seeded synthetic inputs for the Engram forward path (see :mod:`synth.inputs`)."""
from .inputs import *  # noqa: F401,F403
