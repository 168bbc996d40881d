"""CPU oracle of the DFlash 2 drafter pass (test infrastructure only; see ``dflash_oracle``)."""
